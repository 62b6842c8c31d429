"""The C-ABI library loads and exports every entry point include/moe.h declares, and its
host-side argument checks answer before anything reaches a GPU (CPU only)."""

import ctypes
import os
import re

import pytest

from top_routing_grouped_gemm_gb300 import build as B
from top_routing_grouped_gemm_gb300 import moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()


def declared_functions():
    names = set()
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(moe_\w+)\s*\(", src))
    return sorted(names)


def test_every_declared_symbol_is_exported():
    L = ctypes.CDLL(moe.LIB_PATH)
    names = declared_functions()
    assert len(names) >= 17
    for n in names:
        assert hasattr(L, n), n
    assert sorted(moe.exported_symbols()) == names


def test_status_strings_and_version():
    assert moe.moe_status_string(0) == "MOE_OK"
    for s in range(1, 7):
        assert moe.moe_status_string(s).startswith(moe.STATUS_NAMES[s])
    assert moe.moe_version() >= 10000


def _call(name, *args):
    f = getattr(moe.lib(), name)
    return f(*args)


P_OK = moe.Problem(T=64, d=128, E=16, k=4, F=128)
FAKE = 0x10000  # never dereferenced: every call below fails its host checks first


@pytest.mark.parametrize("prob, status", [
    (moe.Problem(T=0, d=128, E=16, k=4, F=128), moe.STATUS_NAMES.get(1)),
    (moe.Problem(T=64, d=100, E=16, k=4, F=128), moe.STATUS_NAMES.get(2)),
    (moe.Problem(T=64, d=128, E=16, k=33, F=128), moe.STATUS_NAMES.get(2)),
    (moe.Problem(T=64, d=128, E=4, k=8, F=128), moe.STATUS_NAMES.get(2)),
    (moe.Problem(T=64, d=128, E=2048, k=8, F=128), moe.STATUS_NAMES.get(2)),
    (moe.Problem(T=64, d=128, E=16, k=4, F=128, r=12), moe.STATUS_NAMES.get(2)),
    (moe.Problem(T=64, d=128, E=16, k=4, F=96), moe.STATUS_NAMES.get(2)),
])
def test_bad_problems_rejected(prob, status):
    st = _call("moe_combine", prob.c(), FAKE, FAKE, FAKE, None)
    assert moe.STATUS_NAMES[st] == status
    assert moe.moe_route_workspace_size(prob) == 0


def test_null_pointers_rejected():
    assert _call("moe_combine", P_OK.c(), None, FAKE, FAKE, None) == 1
    assert _call("moe_route", P_OK.c(), FAKE, None, None, FAKE, FAKE, FAKE, None, FAKE, 1 << 30,
                 None, None) == 1
    assert _call("moe_dispatch", P_OK.c(), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE,
                 1 << 30, None, None) == 1


def test_noalloc_dispatch_follows_moe_dispatch_argument_rules():
    # non-positive sizes: the same MOE_ERR_INVALID_ARG as moe_dispatch, nothing enqueued
    bad = moe.Problem(T=0, d=128, E=16, k=4, F=128)
    args = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None)
    assert _call("moe_dispatch_noalloc", bad.c(), *args) == 1
    assert _call("moe_dispatch", bad.c(), *args[:8], FAKE, 1 << 30, None, None) == 1
    # x_perm without x is rejected by both
    assert _call("moe_dispatch_noalloc", P_OK.c(), FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE,
                 FAKE, None, None) == 1
    # a null index map is rejected
    assert _call("moe_dispatch_noalloc", P_OK.c(), FAKE, None, FAKE, FAKE, None, FAKE, FAKE,
                 None, None, None) == 1


def test_misaligned_pointers_rejected():
    assert _call("moe_combine", P_OK.c(), FAKE + 2, FAKE, FAKE, None) == 2
    assert _call("moe_route", P_OK.c(), FAKE + 8, FAKE, None, FAKE, FAKE, FAKE, None, FAKE,
                 1 << 30, None, None) == 2


def test_small_workspace_rejected():
    need = moe.moe_route_workspace_size(P_OK)
    assert need > 0
    assert _call("moe_route", P_OK.c(), FAKE, FAKE, None, FAKE, FAKE, FAKE, None, FAKE, need - 1,
                 None, None) == 3
    need = moe.moe_dispatch_workspace_size(P_OK)
    assert _call("moe_dispatch", P_OK.c(), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                 need - 1, None, None) == 3
    assert _call("moe_expert_ffn", P_OK.c(), 256, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                 FAKE, FAKE, None, FAKE, 0, None, None) == 3


def test_workspace_sizes_grow_with_problem():
    a = moe.moe_expert_ffn_workspace_size(moe.Problem(64, 128, 16, 4, 128), 256)
    b = moe.moe_expert_ffn_workspace_size(moe.Problem(64, 128, 16, 4, 128, r=16), 256)
    assert b > a > 0
    assert moe.moe_route_num_partials(moe.Problem(4096, 2048, 896, 16, 512)) == 4096 // 8
