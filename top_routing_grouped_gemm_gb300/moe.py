"""ctypes binding of libmoe.so (the C ABI in include/moe.h).

Each ``moe_*`` function here has the name and the argument order of the C entry point and
only marshals arguments: torch tensors become device pointers, the problem becomes a
``moe_problem`` struct, the current torch stream is passed as the CUDA stream, and a
non-zero status raises :class:`MoEError`.  Every computation happens in the CUDA kernels
of the library.  :func:`layer_forward` / :func:`layer_backward` chain the entry points for
one layer and allocate the outputs with torch (the library itself never allocates).

There is no fallback: if libmoe.so is missing or cannot be loaded, calls raise.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

c_i32 = ctypes.c_int32
c_vp = ctypes.c_void_p
c_sz = ctypes.c_size_t

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT",
                6: "MOE_ERR_BAD_INDEX"}


class MoEError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")


class moe_problem(ctypes.Structure):
    _fields_ = [("T", c_i32), ("d", c_i32), ("E", c_i32), ("k", c_i32), ("F", c_i32),
                ("r", c_i32), ("lora_scale", ctypes.c_float), ("cap_num", c_i32),
                ("cap_den", c_i32)]


class moe_lora(ctypes.Structure):
    _fields_ = [(n, c_vp) for n in ("A_g", "B_g", "A_u", "B_u", "A_d", "B_d")]


class moe_lora_grad(ctypes.Structure):
    _fields_ = [(n, c_vp) for n in ("dA_g", "dB_g", "dA_u", "dB_u", "dA_d", "dB_d")]


class moe_ffn_saved(ctypes.Structure):
    _fields_ = [(n, c_vp) for n in ("a_gate", "a_up", "u_gate", "u_up", "u_down")]


_P = ctypes.POINTER(moe_problem)
_SIGS = {
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_version": (ctypes.c_int, []),
    "moe_route_num_partials": (ctypes.c_int, [_P]),
    "moe_route_workspace_size": (c_sz, [_P]),
    "moe_route": (ctypes.c_int, [_P, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp, c_vp]),
    "moe_route_fused_topk": (ctypes.c_int, [_P, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp, c_vp]),
    "moe_route_from_logits": (ctypes.c_int, [_P, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "moe_dispatch_workspace_size": (c_sz, [_P]),
    "moe_dispatch": (ctypes.c_int, [_P, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp, c_vp]),
    "moe_dispatch_noalloc": (ctypes.c_int, [_P, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "moe_route_alternatives": (ctypes.c_int, [_P, c_vp, c_i32, c_vp, c_vp]),
    "moe_dispatch_remap_workspace_size": (c_sz, [_P, c_i32]),
    "moe_dispatch_remap": (ctypes.c_int, [_P, c_vp, c_vp, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp,
                                          c_vp, c_vp, c_vp, c_vp, c_sz, c_vp, c_vp]),
    "moe_dispatch_ep": (ctypes.c_int, [_P, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                       c_vp, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp, c_vp]),
    "moe_expert_counts": (ctypes.c_int, [_P, c_vp, c_vp, c_vp, c_vp]),
    "moe_ep_regroup": (ctypes.c_int, [c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32,
                                      ctypes.c_int64, c_vp, c_vp, c_vp, c_vp]),
    "moe_expert_ffn_workspace_size": (c_sz, [_P, c_i32]),
    "moe_expert_ffn": (ctypes.c_int, [_P, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                      ctypes.POINTER(moe_lora), c_vp, c_vp,
                                      ctypes.POINTER(moe_ffn_saved), c_vp, c_sz, c_vp, c_vp]),
    "moe_expert_ffn_gather": (ctypes.c_int, [_P, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                             ctypes.POINTER(moe_lora), c_vp, c_vp,
                                             ctypes.POINTER(moe_ffn_saved), c_vp, c_sz, c_vp, c_vp]),
    "moe_expert_ffn_combine_workspace_size": (c_sz, [_P, c_i32]),
    "moe_expert_ffn_combine": (ctypes.c_int, [_P, c_i32, c_vp, c_i32, c_vp, c_vp, c_vp, c_vp,
                                              c_vp, c_vp, c_vp, ctypes.POINTER(moe_lora), c_vp,
                                              c_vp, c_vp, ctypes.POINTER(moe_ffn_saved), c_vp,
                                              c_sz, c_vp, c_vp]),
    "moe_combine": (ctypes.c_int, [_P, c_vp, c_vp, c_vp, c_vp]),
    "moe_aux_loss_workspace_size": (c_sz, [_P]),
    "moe_aux_loss": (ctypes.c_int, [_P, c_vp, c_vp, c_i32, c_vp, c_vp, c_sz, c_vp]),
    "moe_combine_bwd": (ctypes.c_int, [_P, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "moe_dispatch_route_bwd": (ctypes.c_int, [_P, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "moe_expert_ffn_bwd_workspace_size": (c_sz, [_P, c_i32]),
    "moe_expert_ffn_bwd": (ctypes.c_int, [_P, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp,
                                          ctypes.POINTER(moe_lora), ctypes.POINTER(moe_ffn_saved),
                                          c_vp, c_vp, c_vp, ctypes.POINTER(moe_lora_grad),
                                          c_vp, c_vp, c_vp,
                                          c_vp, c_sz, c_vp, c_vp]),
    "moe_dispatch_bwd": (ctypes.c_int, [_P, c_vp, c_vp, c_vp, c_vp]),
    "moe_route_bwd": (ctypes.c_int, [_P, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "moe_gdr_workspace_size": (c_sz, [c_i32, c_i32, c_i32, c_i32, c_i32]),
    "moe_gdr_forward": (ctypes.c_int, [c_i32, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp,
                                       c_vp, c_vp, ctypes.c_float, c_vp, c_vp, c_vp, c_vp, c_vp,
                                       c_sz, c_vp]),
    "moe_gdr_device_status": (ctypes.c_int, [ctypes.POINTER(c_i32), c_vp]),
    "moe_gdr_backward_workspace_size": (c_sz, [c_i32, c_i32, c_i32, c_i32, c_i32]),
    "moe_gdr_backward": (ctypes.c_int, [c_i32, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp,
                                        c_vp, ctypes.c_float, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                        c_vp, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp]),
    "moe_set_kernel_events": (ctypes.c_int, [ctypes.c_int, c_vp, c_vp]),
    "moe_launch_count": (ctypes.c_longlong, []),
    "moe_selftest_wait_timeout": (ctypes.c_int, [c_vp, c_i32, c_vp]),
}

KERNEL_IDS = {"router_gemm": 0, "topk": 1, "dispatch": 2, "gateup_gemm": 3, "down_gemm": 4,
              "combine": 5, "bwd_dh_gemm": 6, "bwd_dx_gemm": 7, "wgrad": 8, "gdr_chunk": 9,
              "gdr_scan": 10, "gdr_bwd": 11, "combine_bwd": 12, "dispatch_route_bwd": 13,
              "gdr_bwd_factors": 14, "gdr_bwd_scan": 15}

_lib = None


def lib():
    """Load libmoe.so once; raise if it is missing (there is no fallback path)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run top_routing_grouped_gemm_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def exported_symbols():
    return list(_SIGS)


# ----------------------------------------------------------------------------- marshalling

@dataclass
class Problem:
    T: int
    d: int
    E: int
    k: int
    F: int
    r: int = 0
    lora_scale: float = 0.0
    cap_num: int = 0
    cap_den: int = 0

    def c(self):
        return ctypes.byref(moe_problem(self.T, self.d, self.E, self.k, self.F, self.r,
                                        self.lora_scale, self.cap_num, self.cap_den))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(name, status):
    if status != MOE_OK:
        raise MoEError(name, status)


def _lora(lora):
    if lora is None:
        return None
    return ctypes.byref(moe_lora(*[_ptr(lora[n]) for n in ("A_g", "B_g", "A_u", "B_u", "A_d", "B_d")]))


def _saved(saved):
    if saved is None:
        return None
    return ctypes.byref(moe_ffn_saved(*[_ptr(saved.get(n)) for n in
                                        ("a_gate", "a_up", "u_gate", "u_up", "u_down")]))


def _grads(grads):
    if grads is None:
        return None
    return ctypes.byref(moe_lora_grad(*[_ptr(grads.get(n)) for n in
                                        ("dA_g", "dB_g", "dA_u", "dB_u", "dA_d", "dB_d")]))


def _ws(t):
    return (_ptr(t), 0 if t is None else t.numel() * t.element_size())


# ----------------------------------------------------------------------------- entry points

def moe_status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def moe_version() -> int:
    return lib().moe_version()


def moe_route_num_partials(p: Problem) -> int:
    return lib().moe_route_num_partials(p.c())


def moe_route_workspace_size(p: Problem) -> int:
    return lib().moe_route_workspace_size(p.c())


def moe_route(p, x, w_router, bias, topk_idx, topk_gate, prob_partials, logits, workspace,
              dev_status=None, stream=None):
    wp, wn = _ws(workspace)
    _check("moe_route", lib().moe_route(p.c(), _ptr(x), _ptr(w_router), _ptr(bias),
                                        _ptr(topk_idx), _ptr(topk_gate), _ptr(prob_partials),
                                        _ptr(logits), wp, wn, _ptr(dev_status), _stream(stream)))


def moe_route_fused_topk(p, x, w_router, bias, topk_idx, topk_gate, prob_partials, logits,
                         workspace, dev_status=None, stream=None):
    wp, wn = _ws(workspace)
    _check("moe_route_fused_topk",
           lib().moe_route_fused_topk(p.c(), _ptr(x), _ptr(w_router), _ptr(bias),
                                      _ptr(topk_idx), _ptr(topk_gate), _ptr(prob_partials),
                                      _ptr(logits), wp, wn, _ptr(dev_status), _stream(stream)))


def moe_route_from_logits(p, logits, topk_idx, topk_gate, prob_partials, dev_status=None,
                          stream=None):
    _check("moe_route_from_logits",
           lib().moe_route_from_logits(p.c(), _ptr(logits), _ptr(topk_idx), _ptr(topk_gate),
                                       _ptr(prob_partials), _ptr(dev_status), _stream(stream)))


def moe_dispatch_workspace_size(p: Problem) -> int:
    return lib().moe_dispatch_workspace_size(p.c())


def moe_dispatch(p, topk_idx, x, counts, offsets, slot_row, row_slot, n_kept_dropped, x_perm,
                 workspace, dev_status=None, stream=None):
    wp, wn = _ws(workspace)
    _check("moe_dispatch", lib().moe_dispatch(p.c(), _ptr(topk_idx), _ptr(x), _ptr(counts),
                                              _ptr(offsets), _ptr(slot_row), _ptr(row_slot),
                                              _ptr(n_kept_dropped), _ptr(x_perm), wp, wn,
                                              _ptr(dev_status), _stream(stream)))


def moe_dispatch_noalloc(p, topk_idx, x, counts, offsets, slot_row, row_slot, n_kept_dropped,
                         x_perm, dev_status=None, stream=None):
    """moe_dispatch with the library's built-in scratch instead of a caller workspace."""
    _check("moe_dispatch_noalloc",
           lib().moe_dispatch_noalloc(p.c(), _ptr(topk_idx), _ptr(x), _ptr(counts), _ptr(offsets),
                                      _ptr(slot_row), _ptr(row_slot), _ptr(n_kept_dropped),
                                      _ptr(x_perm), _ptr(dev_status), _stream(stream)))


def moe_route_alternatives(p, logits, n_alt, alt_idx, stream=None):
    _check("moe_route_alternatives",
           lib().moe_route_alternatives(p.c(), _ptr(logits), n_alt, _ptr(alt_idx),
                                        _stream(stream)))


def moe_dispatch_remap_workspace_size(p: Problem, rounds: int) -> int:
    return lib().moe_dispatch_remap_workspace_size(p.c(), rounds)


def moe_dispatch_remap(p, topk_idx, alt_idx, rounds, x, counts, offsets, slot_row, row_slot,
                       slot_expert, n_kept_dropped, x_perm, workspace, dev_status=None,
                       stream=None):
    wp, wn = _ws(workspace)
    _check("moe_dispatch_remap",
           lib().moe_dispatch_remap(p.c(), _ptr(topk_idx), _ptr(alt_idx), rounds, _ptr(x),
                                    _ptr(counts), _ptr(offsets), _ptr(slot_row), _ptr(row_slot),
                                    _ptr(slot_expert), _ptr(n_kept_dropped), _ptr(x_perm), wp, wn,
                                    _ptr(dev_status), _stream(stream)))


def moe_dispatch_ep(p, capacity, topk_idx, topk_gate, x, pos_base, counts, offsets, slot_row,
                    row_slot, n_kept_dropped, x_perm, gate_perm, workspace, dev_status=None,
                    stream=None):
    """capacity: C of the whole batch (None or negative: no limit)."""
    wp, wn = _ws(workspace)
    C = -1 if capacity is None or capacity < 0 else int(capacity)
    _check("moe_dispatch_ep",
           lib().moe_dispatch_ep(p.c(), C, _ptr(topk_idx), _ptr(topk_gate), _ptr(x), _ptr(pos_base),
                                 _ptr(counts), _ptr(offsets), _ptr(slot_row), _ptr(row_slot),
                                 _ptr(n_kept_dropped), _ptr(x_perm), _ptr(gate_perm), wp, wn,
                                 _ptr(dev_status), _stream(stream)))


def moe_expert_counts(p, topk_idx, counts, dev_status=None, stream=None):
    _check("moe_expert_counts", lib().moe_expert_counts(p.c(), _ptr(topk_idx), _ptr(counts),
                                                        _ptr(dev_status), _stream(stream)))


def moe_ep_regroup(src, gate_src, kept, n_sources, n_local_experts, d, to_expert_major,
                   rows_total, dst, gate_dst, expert_offsets, stream=None):
    _check("moe_ep_regroup",
           lib().moe_ep_regroup(_ptr(src), _ptr(gate_src), _ptr(kept), n_sources,
                                n_local_experts, d, 1 if to_expert_major else 0, rows_total,
                                _ptr(dst), _ptr(gate_dst), _ptr(expert_offsets),
                                _stream(stream)))


def moe_expert_ffn_workspace_size(p: Problem, rows_max: int) -> int:
    return lib().moe_expert_ffn_workspace_size(p.c(), rows_max)


def moe_expert_ffn(p, rows_max, x_perm, offsets, row_slot, topk_gate, w_gate, w_up, w_down,
                   lora, h, y_perm, saved, workspace, dev_status=None, stream=None):
    wp, wn = _ws(workspace)
    _check("moe_expert_ffn",
           lib().moe_expert_ffn(p.c(), rows_max, _ptr(x_perm), _ptr(offsets), _ptr(row_slot),
                                _ptr(topk_gate), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                                _lora(lora), _ptr(h), _ptr(y_perm), _saved(saved), wp, wn,
                                _ptr(dev_status), _stream(stream)))


def moe_expert_ffn_gather(p, rows_max, x, offsets, row_slot, topk_gate, w_gate, w_up, w_down,
                          lora, h, y_perm, saved, workspace, dev_status=None, stream=None):
    wp, wn = _ws(workspace)
    _check("moe_expert_ffn_gather",
           lib().moe_expert_ffn_gather(p.c(), rows_max, _ptr(x), _ptr(offsets), _ptr(row_slot),
                                       _ptr(topk_gate), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                                       _lora(lora), _ptr(h), _ptr(y_perm), _saved(saved), wp, wn,
                                       _ptr(dev_status), _stream(stream)))


def moe_expert_ffn_combine_workspace_size(p: Problem, rows_max: int) -> int:
    return lib().moe_expert_ffn_combine_workspace_size(p.c(), rows_max)


def moe_expert_ffn_combine(p, rows_max, a_src, a_is_tokens, offsets, row_slot, slot_row,
                           topk_gate, w_gate, w_up, w_down, lora, h, y_perm, y, saved,
                           workspace, dev_status=None, stream=None):
    wp, wn = _ws(workspace)
    _check("moe_expert_ffn_combine",
           lib().moe_expert_ffn_combine(p.c(), rows_max, _ptr(a_src), 1 if a_is_tokens else 0,
                                        _ptr(offsets), _ptr(row_slot), _ptr(slot_row),
                                        _ptr(topk_gate), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                                        _lora(lora), _ptr(h), _ptr(y_perm), _ptr(y),
                                        _saved(saved), wp, wn, _ptr(dev_status),
                                        _stream(stream)))


def moe_combine(p, y_perm, slot_row, y, stream=None):
    _check("moe_combine", lib().moe_combine(p.c(), _ptr(y_perm), _ptr(slot_row), _ptr(y),
                                            _stream(stream)))


def moe_aux_loss_workspace_size(p: Problem) -> int:
    return lib().moe_aux_loss_workspace_size(p.c())


def moe_aux_loss(p, counts, prob_partials, n_partials, aux_out, workspace, stream=None):
    wp, wn = _ws(workspace)
    _check("moe_aux_loss", lib().moe_aux_loss(p.c(), _ptr(counts), _ptr(prob_partials),
                                              n_partials, _ptr(aux_out), wp, wn, _stream(stream)))


def moe_combine_bwd(p, dy, y_perm, slot_row, topk_gate, dz_perm, dgate, stream=None):
    _check("moe_combine_bwd", lib().moe_combine_bwd(p.c(), _ptr(dy), _ptr(y_perm), _ptr(slot_row),
                                                    _ptr(topk_gate), _ptr(dz_perm), _ptr(dgate),
                                                    _stream(stream)))


def moe_expert_ffn_bwd_workspace_size(p: Problem, rows_max: int) -> int:
    return lib().moe_expert_ffn_bwd_workspace_size(p.c(), rows_max)


def moe_expert_ffn_bwd(p, rows_max, x_perm, offsets, w_gate, w_up, w_down, lora, saved, h,
                       dz_perm, dx_perm, grads, workspace, dev_status=None, stream=None,
                       row_slot=None, topk_gate=None, dgate=None):
    wp, wn = _ws(workspace)
    _check("moe_expert_ffn_bwd",
           lib().moe_expert_ffn_bwd(p.c(), rows_max, _ptr(x_perm), _ptr(offsets), _ptr(w_gate),
                                    _ptr(w_up), _ptr(w_down), _lora(lora), _saved(saved), _ptr(h),
                                    _ptr(dz_perm), _ptr(dx_perm), _grads(grads), _ptr(row_slot),
                                    _ptr(topk_gate), _ptr(dgate), wp, wn, _ptr(dev_status),
                                    _stream(stream)))


def moe_dispatch_route_bwd(p, dx_perm, slot_row, topk_idx, topk_gate, dgate, w_router, dx,
                           stream=None):
    _check("moe_dispatch_route_bwd",
           lib().moe_dispatch_route_bwd(p.c(), _ptr(dx_perm), _ptr(slot_row), _ptr(topk_idx),
                                        _ptr(topk_gate), _ptr(dgate), _ptr(w_router), _ptr(dx),
                                        _stream(stream)))


def moe_dispatch_bwd(p, dx_perm, slot_row, dx, stream=None):
    _check("moe_dispatch_bwd", lib().moe_dispatch_bwd(p.c(), _ptr(dx_perm), _ptr(slot_row),
                                                      _ptr(dx), _stream(stream)))


def moe_route_bwd(p, topk_idx, topk_gate, dgate, w_router, dx, stream=None):
    _check("moe_route_bwd", lib().moe_route_bwd(p.c(), _ptr(topk_idx), _ptr(topk_gate),
                                                _ptr(dgate), _ptr(w_router), _ptr(dx),
                                                _stream(stream)))


# ---- gated delta-rule linear attention (include/linear_attention.h)

def moe_gdr_workspace_size(B, T, H, dk, dv) -> int:
    return lib().moe_gdr_workspace_size(B, T, H, dk, dv)


def moe_gdr_forward(B, T, H, dk, dv, q, k, v, beta, g, S0, scale, o, S_T, S_chunks, workspace,
                    stream=None, W_chunks=None):
    wp, wn = _ws(workspace)
    _check("moe_gdr_forward",
           lib().moe_gdr_forward(B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
                                 _ptr(S0), scale, _ptr(o), _ptr(S_T), _ptr(S_chunks),
                                 _ptr(W_chunks), wp, wn, _stream(stream)))


def moe_gdr_device_status(stream=None) -> int:
    """Waits for ``stream``; the first status a linear-attention kernel recorded since the
    previous call (0: none), cleared."""
    st = c_i32(0)
    _check("moe_gdr_device_status", lib().moe_gdr_device_status(ctypes.byref(st), _stream(stream)))
    return int(st.value)


def moe_gdr_backward_workspace_size(B, T, H, dk, dv) -> int:
    return lib().moe_gdr_backward_workspace_size(B, T, H, dk, dv)


def moe_gdr_backward(B, T, H, dk, dv, q, k, v, beta, g, scale, d_o, dS_T, S_chunks, dq, dk_,
                     dv_, dbeta, dg, dS0, workspace, stream=None, W_chunks=None):
    wp, wn = _ws(workspace)
    _check("moe_gdr_backward",
           lib().moe_gdr_backward(B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
                                  scale, _ptr(d_o), _ptr(dS_T), _ptr(S_chunks), _ptr(W_chunks),
                                  _ptr(dq), _ptr(dk_), _ptr(dv_), _ptr(dbeta), _ptr(dg), _ptr(dS0),
                                  wp, wn, _stream(stream)))


def moe_set_kernel_events(kernel, before, after):
    """Record torch.cuda.Event ``before``/``after`` around the next launches of ``kernel``
    (a name of KERNEL_IDS); ``None`` stops recording."""
    kid = KERNEL_IDS[kernel] if isinstance(kernel, str) else int(kernel)
    hb = before.cuda_event if before is not None else None
    ha = after.cuda_event if after is not None else None
    if (before is not None and not hb) or (after is not None and not ha):
        raise ValueError("record each torch.cuda.Event once before handing it to the library")
    _check("moe_set_kernel_events", lib().moe_set_kernel_events(kid, hb, ha))


def moe_launch_count() -> int:
    return lib().moe_launch_count()


def moe_selftest_wait_timeout(dev_status, timeout_ms, stream=None):
    _check("moe_selftest_wait_timeout",
           lib().moe_selftest_wait_timeout(_ptr(dev_status), timeout_ms, _stream(stream)))


# ----------------------------------------------------------------------------- layer helpers

def problem_of(cfg) -> Problem:
    return Problem(cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.r, cfg.lora_scale, cfg.cap_num,
                   cfg.cap_den)


def _empty(shape, dtype, device):
    return torch.empty(shape, dtype=dtype, device=device)


def _bytes(n, device):
    return torch.empty(max(int(n), 1), dtype=torch.uint8, device=device)


class LayerBuffers:
    """Every device buffer one forward (and, with ``train=True``, one backward) of the layer
    uses, allocated once with torch and reused across calls."""

    def __init__(self, p: Problem, device="cuda", train=False, keep_logits=True,
                 remap_rounds=0):
        dev = torch.device(device)
        T, d, E, k, F, r = p.T, p.d, p.E, p.k, p.F, p.r
        N = T * k
        self.p = p
        self.rows_max = N
        self.remap_rounds = remap_rounds
        keep_logits = keep_logits or remap_rounds > 0   # the alternatives are read from them
        self.logits = _empty((T, E), torch.float32, dev) if keep_logits else None
        if remap_rounds:
            self.alt_idx = _empty((T, remap_rounds * k), torch.int32, dev)
            self.slot_expert = _empty((N,), torch.int32, dev)
            self.ws_remap = _bytes(moe_dispatch_remap_workspace_size(p, remap_rounds), dev)
        self.topk_idx = _empty((T, k), torch.int32, dev)
        self.topk_gate = _empty((T, k), torch.float32, dev)
        self.n_partials = moe_route_num_partials(p)
        self.partials = _empty((self.n_partials, E), torch.float32, dev)
        self.counts = _empty((E,), torch.int32, dev)
        self.offsets = _empty((E + 1,), torch.int32, dev)
        self.slot_row = _empty((N,), torch.int32, dev)
        self.row_slot = _empty((N,), torch.int32, dev)
        self.n_kept_dropped = _empty((2,), torch.int32, dev)
        self.x_perm = _empty((N, d), torch.bfloat16, dev)
        self.h = _empty((N, F), torch.bfloat16, dev)
        self.y_perm = _empty((N, d), torch.bfloat16, dev)
        self.y = _empty((T, d), torch.bfloat16, dev)
        self.aux = _empty((1,), torch.float32, dev)
        self.dev_status = torch.zeros((1,), dtype=torch.int32, device=dev)
        self.ws_route = _bytes(moe_route_workspace_size(p), dev)
        self.ws_dispatch = _bytes(moe_dispatch_workspace_size(p), dev)
        self.ws_ffn = _bytes(moe_expert_ffn_combine_workspace_size(p, N), dev)
        self.ws_aux = _bytes(moe_aux_loss_workspace_size(p), dev)
        self.saved = None
        self.train = train
        if train:
            self.saved = {"a_gate": _empty((N, F), torch.bfloat16, dev),
                          "a_up": _empty((N, F), torch.bfloat16, dev)}
            if r:
                for n in ("u_gate", "u_up", "u_down"):
                    self.saved[n] = _empty((N, r), torch.bfloat16, dev)
            self.dz_perm = _empty((N, d), torch.bfloat16, dev)
            self.dgate = _empty((T, k), torch.float32, dev)
            self.dx_perm = _empty((N, d), torch.bfloat16, dev)
            self.dx = _empty((T, d), torch.float32, dev)
            self.ws_bwd = _bytes(moe_expert_ffn_bwd_workspace_size(p, N), dev)
            self.grads = None
            if r:
                self.grads = {"dA_g": _empty((E, r, d), torch.float32, dev),
                              "dB_g": _empty((E, F, r), torch.float32, dev),
                              "dA_u": _empty((E, r, d), torch.float32, dev),
                              "dB_u": _empty((E, F, r), torch.float32, dev),
                              "dA_d": _empty((E, r, F), torch.float32, dev),
                              "dB_d": _empty((E, d, r), torch.float32, dev)}


# The fused permute gathers token rows inside the expert GEMM; it pays off while the token
# matrix stays resident in the 129 MB L2 (the gathers then hit L2), not beyond.
FUSED_PERMUTE_MAX_X_BYTES = 48 << 20


def fused_permute_default(p: Problem, train: bool) -> bool:
    return (not train) and p.T * p.d * 2 <= FUSED_PERMUTE_MAX_X_BYTES


def layer_forward(buf: LayerBuffers, x, w_router, bias, w_gate, w_up, w_down, lora=None,
                  stream=None, gather=None, fuse_combine=False):
    """route -> dispatch -> experts -> combine -> aux, all enqueued on one stream.

    gather=True fuses the permute into the expert GEMMs (moe_expert_ffn_gather: dispatch
    writes only the index maps and the GEMM copies token rows of x into its operand tiles);
    gather=False writes x_perm.  The default fuses when x fits well in L2 and no backward
    (which reads x_perm) will follow."""
    p = buf.p
    if gather is None:
        gather = fused_permute_default(p, buf.train)
    moe_route(p, x, w_router, bias, buf.topk_idx, buf.topk_gate, buf.partials, buf.logits,
              buf.ws_route, buf.dev_status, stream)
    if buf.remap_rounds:
        # overflowing slots move to the token's next preferences instead of being dropped
        R = buf.remap_rounds
        moe_route_alternatives(p, buf.logits, R * p.k, buf.alt_idx, stream)
        moe_dispatch_remap(p, buf.topk_idx, buf.alt_idx, R, None if gather else x, buf.counts,
                           buf.offsets, buf.slot_row, buf.row_slot, buf.slot_expert,
                           buf.n_kept_dropped, None if gather else buf.x_perm, buf.ws_remap,
                           buf.dev_status, stream)
    else:
        moe_dispatch(p, buf.topk_idx, None if gather else x, buf.counts, buf.offsets,
                     buf.slot_row, buf.row_slot, buf.n_kept_dropped,
                     None if gather else buf.x_perm, buf.ws_dispatch, buf.dev_status, stream)
    if fuse_combine:
        # unpermute inside the down GEMM's epilogue (same bits as the separate combine)
        moe_expert_ffn_combine(p, buf.rows_max, x if gather else buf.x_perm, gather,
                               buf.offsets, buf.row_slot, buf.slot_row, buf.topk_gate, w_gate,
                               w_up, w_down, lora, buf.h, buf.y_perm, buf.y, buf.saved,
                               buf.ws_ffn, buf.dev_status, stream)
    else:
        ffn = moe_expert_ffn_gather if gather else moe_expert_ffn
        ffn(p, buf.rows_max, x if gather else buf.x_perm, buf.offsets, buf.row_slot,
            buf.topk_gate, w_gate, w_up, w_down, lora, buf.h, buf.y_perm, buf.saved, buf.ws_ffn,
            buf.dev_status, stream)
        moe_combine(p, buf.y_perm, buf.slot_row, buf.y, stream)
    moe_aux_loss(p, buf.counts, buf.partials, buf.n_partials, buf.aux, buf.ws_aux, stream)
    return buf.y


def layer_backward(buf: LayerBuffers, dy, x, w_router, w_gate, w_up, w_down, lora=None,
                   stream=None):
    """Gradient of <dy, y> for the forward last run on ``buf`` (which must have been built
    with train=True): combine backward (dz_perm) -> expert backward (dx_perm, LoRA grads, and
    the gate gradients from its dh product) -> dispatch and router backward in one pass (the
    expert path and the gate path of dx)."""
    p = buf.p
    assert buf.train, "LayerBuffers(train=True) keeps what the backward needs"
    moe_combine_bwd(p, dy, None, buf.slot_row, buf.topk_gate, buf.dz_perm, buf.dgate, stream)
    moe_expert_ffn_bwd(p, buf.rows_max, buf.x_perm, buf.offsets, w_gate, w_up, w_down, lora,
                       buf.saved, buf.h, buf.dz_perm, buf.dx_perm, buf.grads, buf.ws_bwd,
                       buf.dev_status, stream, row_slot=buf.row_slot, topk_gate=buf.topk_gate,
                       dgate=buf.dgate)
    moe_dispatch_route_bwd(p, buf.dx_perm, buf.slot_row, buf.topk_idx, buf.topk_gate,
                           buf.dgate, w_router, buf.dx, stream)
    return buf.dx
