"""Expert-parallel (EP) forward of the MoE layer: the experts split over P ranks, every rank
routing its own tokens, with the exchange of "Trillion-Parameter MoE Model Training
Adaptation: Full-Stack Optimization Practices", section 3 "Communication" (tokens permuted
by routing result are sent with an All-to-All to the GPUs hosting their experts, computed in
grouped GEMMs, then unpermuted and returned), section 4.1 (expert parallelism: the 896
experts divided evenly, E/P contiguous experts per rank, placed statically) and section 4.3
(compute-communication overlap: chunk i is transferred while chunk i-1 is computed,
pipelining dispatch and expert computation).

One step on rank r of P, with El = E/P local experts (experts r*El .. r*El+El-1) and the
rank's T tokens cut into n_chunks chunks:

  1. route the rank's T tokens with the replicated router             moe_route
  2. per-chunk expert slot counts                                      moe_expert_counts
  X1. all-gather of the counts -> cnt[P, n_chunks, E]
  3. plan (host, ``plan_exchange``): global arrival order is ranks in order, then chunks,
     then tokens, so part (s, c)'s slots of expert e start at base[s, c, e] = the sum of
     cnt over the parts before it; with a capacity C a slot at local position pos is kept
     iff base + pos < C, so kept[s, c, e] = clamp(C - base[s, c, e], 0, cnt[s, c, e])
  then, per chunk c (chunk c + 1's dispatch and transfer overlap chunk c's experts):
  4. dispatch with that base: x_perm is expert-major over all E experts, so the rows for
     rank d (d's experts) are one contiguous slice; each row's gate travels with it
                                                                       moe_dispatch_ep
  X2. all-to-all-v of the rows and their gates (send split d: rows of d's experts;
     receive split s: sum of kept[s, c, mine])
  5. regroup the received rows source-major -> expert-major            moe_ep_regroup
  6. grouped expert GEMMs on the local experts, gate-scaled            moe_expert_ffn
  7. regroup the results expert-major -> source-major                  moe_ep_regroup
  X3. the reverse all-to-all-v: every rank gets its rows back in its own x_perm order
  8. combine the chunk's tokens in rank order of their slots           moe_combine
  aux: counts summed over ranks and chunks, probability partials all-gathered
                                                                       moe_aux_loss

With every rank's tokens taken in rank order as one batch, the result is the single-device
layer's on that batch: the same routing, the same kept and dropped slots (capacity is decided
in global arrival order), and, row for row, the same expert products.  With P = 1 and
several chunks this is the single-device layer with its dispatch pipelined against the
expert GEMMs of the previous chunk.

The exchanges are pluggable: :class:`DistExchange` runs them as torch.distributed
collectives (NCCL on GPUs, gloo on CPU), one rank per process; :class:`LocalExchange` holds
all P ranks in one process and moves the tensors directly, which runs the ranks' steps in
lockstep on one device (no kernel ever waits for another rank).  The per-rank compute is a
backend object; :class:`CudaBackend` is the CUDA path through the C ABI.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from . import moe


# ----------------------------------------------------------------------------- host plan

@dataclass
class ExchangePlan:
    """Host-side bookkeeping of one step's exchange (all arrays numpy int64)."""
    P: int
    E: int
    El: int
    C: int | None
    cnt: np.ndarray    # [P, E] slots routed to each expert by each rank (before drops)
    base: np.ndarray   # [P, E] slots of the expert that arrived on earlier ranks
    kept: np.ndarray   # [P, E] slots kept (within capacity in global arrival order)

    def owner_range(self, d):
        return d * self.El, (d + 1) * self.El

    def send_splits(self, r):
        """Rows rank r sends to each rank d (its kept rows of d's experts)."""
        return [int(self.kept[r, d * self.El:(d + 1) * self.El].sum()) for d in range(self.P)]

    def recv_splits(self, r):
        """Rows rank r receives from each source s (s's kept rows of r's experts)."""
        lo, hi = self.owner_range(r)
        return [int(self.kept[s, lo:hi].sum()) for s in range(self.P)]

    def kept_local(self, r):
        """[P, El] kept rows of (source, local expert) for rank r's experts."""
        lo, hi = self.owner_range(r)
        return self.kept[:, lo:hi]

    def n_kept(self, r):
        return int(self.kept[r].sum())


def capacity(T_total: int, k: int, E: int, cap_num: int, cap_den: int):
    """ceil(cf * T * k / E) over the whole batch of all ranks (None: unlimited)."""
    if cap_den == 0:
        return None
    return -(-(cap_num * T_total * k) // (cap_den * E))


def plan_exchange(cnt, C, base=None) -> ExchangePlan:
    """Arrival bases, kept counts and split sizes from the all-gathered counts [P, E].
    ``base`` [P, E] overrides the bases (parts of a larger batch); by default rank s's
    slots of an expert follow those of ranks 0 .. s-1."""
    cnt = np.asarray(cnt, dtype=np.int64)
    P, E = cnt.shape
    if E % P:
        raise ValueError(f"{E} experts do not split evenly over {P} ranks")
    if base is None:
        base = np.zeros_like(cnt)
        base[1:] = np.cumsum(cnt, axis=0)[:-1]
    base = np.asarray(base, dtype=np.int64)
    if C is None:
        kept = cnt.copy()
    else:
        kept = np.clip(C - base, 0, cnt)
    return ExchangePlan(P=P, E=E, El=E // P, C=C, cnt=cnt, base=base, kept=kept)


def plan_chunks(cnt, C):
    """One plan per chunk from the counts [P, n_chunks, E]: the global arrival order is
    ranks, then chunks, then tokens."""
    cnt = np.asarray(cnt, dtype=np.int64)
    P, n, E = cnt.shape
    flat = cnt.reshape(P * n, E)
    base = np.zeros_like(flat)
    base[1:] = np.cumsum(flat, axis=0)[:-1]
    base = base.reshape(P, n, E)
    return [plan_exchange(cnt[:, c], C, base[:, c]) for c in range(n)]


def chunk_bounds(T, n_chunks):
    """Token ranges of n_chunks nearly equal chunks (multiples of 8 tokens where possible)."""
    n_chunks = max(1, min(n_chunks, T))
    step = -(-T // n_chunks)
    step = -(-step // 8) * 8 if step > 8 else step
    out, t = [], 0
    while t < T:
        out.append((t, min(T, t + step)))
        t += step
    return out


# ----------------------------------------------------------------------------- exchanges

class DistExchange:
    """The exchanges as torch.distributed collectives: one rank per process (NCCL for CUDA
    tensors, gloo for CPU tensors).  Methods take and return lists of one tensor (this
    process's rank), like :class:`LocalExchange`."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.P = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.local_ranks = [self.rank]

    def all_gather(self, ts):
        t = ts[0].contiguous()
        out = [torch.empty_like(t) for _ in range(self.P)]
        self.dist.all_gather(out, t, group=self.group)
        return [torch.stack(out)]

    def all_to_all(self, ts, send_splits, recv_splits):
        t = ts[0]
        out = torch.empty((sum(recv_splits[0]),) + tuple(t.shape[1:]), dtype=t.dtype,
                          device=t.device)
        self.dist.all_to_all_single(out, t.contiguous(), output_split_sizes=recv_splits[0],
                                    input_split_sizes=send_splits[0], group=self.group)
        return [out]


class LocalExchange:
    """All P ranks in one process: the exchanges move tensors between the ranks' lists
    directly (same device), so the P ranks' steps run in lockstep."""

    def __init__(self, P):
        self.P = P
        self.local_ranks = list(range(P))

    def all_gather(self, ts):
        s = torch.stack([t.contiguous() for t in ts])
        return [s for _ in ts]

    def all_to_all(self, ts, send_splits, recv_splits):
        pieces = []
        for s, t in enumerate(ts):
            pieces.append(list(torch.split(t, send_splits[s])))
        out = []
        for d in range(self.P):
            parts = [pieces[s][d] for s in range(self.P)]
            assert [int(x.shape[0]) for x in parts] == list(recv_splits[d])
            out.append(torch.cat(parts) if parts else ts[d][:0])
        return out


# ----------------------------------------------------------------------------- CUDA backend

class CudaBackend:
    """The per-rank steps on the GPU through the C ABI of libmoe.so.  ``streams`` = (main,
    side) pipelines the chunks: dispatch and transfers on the side stream, expert GEMMs on
    the main stream."""

    def __init__(self, device="cuda", pipeline=True):
        self.device = torch.device(device)
        self.pipeline = pipeline and self.device.type == "cuda"

    def _i32(self, n):
        return torch.empty((n,), dtype=torch.int32, device=self.device)

    def route(self, p, x, w_router, bias, st):
        st.topk_idx = torch.empty((p.T, p.k), dtype=torch.int32, device=self.device)
        st.topk_gate = torch.empty((p.T, p.k), dtype=torch.float32, device=self.device)
        st.partials = torch.empty((moe.moe_route_num_partials(p), p.E), dtype=torch.float32,
                                  device=self.device)
        ws = torch.empty(moe.moe_route_workspace_size(p), dtype=torch.uint8, device=self.device)
        moe.moe_route(p, x, w_router, bias, st.topk_idx, st.topk_gate, st.partials, None, ws,
                      st.dev_status)

    def counts(self, p, idx, st):
        c = self._i32(p.E)
        moe.moe_expert_counts(p, idx, c, st.dev_status)
        return c

    def dispatch(self, p, C, idx, gate, x, pos_base, st):
        N = p.T * p.k
        ch = _State()
        ch.pos_base = torch.as_tensor(pos_base, dtype=torch.int32).to(self.device)
        ch.counts = self._i32(p.E)
        ch.offsets = self._i32(p.E + 1)
        ch.slot_row = self._i32(N)
        ch.row_slot = self._i32(N)
        ch.n_kept_dropped = self._i32(2)
        ch.x_perm = torch.empty((N, p.d), dtype=torch.bfloat16, device=self.device)
        ch.gate_perm = torch.empty((N,), dtype=torch.float32, device=self.device)
        ws = torch.empty(moe.moe_dispatch_workspace_size(p), dtype=torch.uint8,
                         device=self.device)
        moe.moe_dispatch_ep(p, C, idx, gate, x, ch.pos_base, ch.counts, ch.offsets,
                            ch.slot_row, ch.row_slot, ch.n_kept_dropped, ch.x_perm,
                            ch.gate_perm, ws, st.dev_status)
        return ch

    def regroup(self, src, gsrc, kept, to_expert, d):
        P, El = kept.shape
        rows = int(kept.sum())
        dst = torch.empty((rows, d), dtype=torch.bfloat16, device=self.device)
        gdst = None if gsrc is None else torch.empty((rows,), dtype=torch.float32,
                                                     device=self.device)
        offs = self._i32(El + 1) if to_expert else None
        kept_dev = torch.as_tensor(np.ascontiguousarray(kept), dtype=torch.int32).to(self.device)
        moe.moe_ep_regroup(src if rows else None, gsrc, kept_dev, P, El, d, to_expert, rows,
                           dst if rows else None, gdst, offs)
        return dst, gdst, offs

    def experts(self, p_loc, x_loc, offsets, gates, w_gate, w_up, w_down, lora, st):
        rows = int(x_loc.shape[0])
        y = torch.empty((max(rows, 1), p_loc.d), dtype=torch.bfloat16, device=self.device)
        if rows == 0:
            return y[:0]
        h = torch.empty((rows, p_loc.F), dtype=torch.bfloat16, device=self.device)
        row_slot = torch.arange(rows, dtype=torch.int32, device=self.device)
        ws = torch.empty(moe.moe_expert_ffn_workspace_size(p_loc, rows), dtype=torch.uint8,
                         device=self.device)
        moe.moe_expert_ffn(p_loc, rows, x_loc, offsets, row_slot, gates, w_gate, w_up, w_down,
                           lora, h, y, None, ws, st.dev_status)
        return y

    def combine(self, p, y_perm, slot_row, y_out, st):
        if y_perm.shape[0] == 0:  # every slot dropped: combine reads no row (y = 0)
            y_perm = torch.empty((1, p.d), dtype=torch.bfloat16, device=self.device)
        moe.moe_combine(p, y_perm, slot_row, y_out)

    def new_output(self, T, d):
        return torch.empty((T, d), dtype=torch.bfloat16, device=self.device)

    def aux(self, p_total, counts_total, partials_all, st):
        aux = torch.empty((1,), dtype=torch.float32, device=self.device)
        ws = torch.empty(moe.moe_aux_loss_workspace_size(p_total), dtype=torch.uint8,
                         device=self.device)
        moe.moe_aux_loss(p_total, counts_total.to(torch.int32).contiguous(),
                         partials_all.contiguous(), int(partials_all.shape[0]), aux, ws)
        return aux


# ----------------------------------------------------------------------------- driver

@dataclass
class EPRank:
    """One rank's inputs and, after :func:`ep_forward`, its outputs and intermediates."""
    rank: int
    x: torch.Tensor                  # [T, d] this rank's tokens
    w_gate: torch.Tensor             # [El, F, d] this rank's experts
    w_up: torch.Tensor               # [El, F, d]
    w_down: torch.Tensor             # [El, d, F]
    lora: dict | None = None         # LoRA factors of this rank's experts, or None
    dev_status: torch.Tensor | None = None
    extra: dict = field(default_factory=dict)


class _State:
    pass


class _NoStream:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def _on(stream):
    return torch.cuda.stream(stream) if stream is not None else _NoStream()


def _sub(p, T):
    return moe.Problem(T=T, d=p.d, E=p.E, k=p.k, F=p.F, r=p.r, lora_scale=p.lora_scale,
                       cap_num=p.cap_num, cap_den=p.cap_den)


def ep_forward(p, ranks, w_router, bias, xchg, backend, n_chunks=1):
    """The EP forward for the ranks this process holds (``xchg.local_ranks``).  ``p`` is the
    per-rank problem (T tokens per rank, all E experts; capacity over the whole batch of
    P * T tokens).  Returns, per local rank, dict(y, aux, plans, state)."""
    P = xchg.P
    if p.E % P:
        raise ValueError(f"{p.E} experts do not split evenly over {P} ranks")
    El = p.E // P
    bounds = chunk_bounds(p.T, n_chunks)
    n = len(bounds)
    pipelined = getattr(backend, "pipeline", False)
    main = torch.cuda.current_stream() if pipelined else None
    side = torch.cuda.Stream() if pipelined else None
    sts = []
    for r in ranks:
        st = _State()
        st.dev_status = r.dev_status if r.dev_status is not None else             torch.zeros((1,), dtype=torch.int32, device=r.x.device)
        backend.route(p, r.x, w_router, bias, st)
        st.cnt = torch.stack([backend.counts(_sub(p, t1 - t0), st.topk_idx[t0:t1], st)
                              for t0, t1 in bounds])
        st.y = backend.new_output(p.T, p.d)
        sts.append(st)
    # X1: counts of every rank and chunk
    cnt_all = xchg.all_gather([st.cnt for st in sts])
    C = capacity(P * p.T, p.k, p.E, p.cap_num, p.cap_den)
    plans = [plan_chunks(c.cpu().numpy(), C) for c in cnt_all]
    p_loc = moe.Problem(T=max(1, p.T * p.k * P), d=p.d, E=El, k=1, F=p.F, r=p.r,
                        lora_scale=p.lora_scale)
    if pipelined:
        side.wait_stream(main)

    def dispatch_and_send(c):
        t0, t1 = bounds[c]
        pc = _sub(p, t1 - t0)
        chs, xs, gs, send, recv = [], [], [], [], []
        with _on(side):
            for i, (r, st) in enumerate(zip(ranks, sts)):
                plan = plans[i][c]
                ch = backend.dispatch(pc, C, st.topk_idx[t0:t1], st.topk_gate[t0:t1],
                                      r.x[t0:t1], plan.base[r.rank], st)
                nk = plan.n_kept(r.rank)
                chs.append(ch)
                xs.append(ch.x_perm[:nk])
                gs.append(ch.gate_perm[:nk])
                send.append(plan.send_splits(r.rank))
                recv.append(plan.recv_splits(r.rank))
            # X2: rows and gates to the ranks holding their experts
            xr = xchg.all_to_all(xs, send, recv)
            gr = xchg.all_to_all(gs, send, recv)
            ev = None
            if pipelined:
                ev = torch.cuda.Event()
                ev.record(side)
                for t in xr + gr:
                    t.record_stream(main)
        return dict(chs=chs, xr=xr, gr=gr, send=send, recv=recv, ev=ev, pc=pc)

    pending = dispatch_and_send(0)
    for c in range(n):
        cur = pending
        if pipelined:
            main.wait_event(cur["ev"])
        y_back = []
        for i, (r, st) in enumerate(zip(ranks, sts)):
            kl = plans[i][c].kept_local(r.rank)
            x_loc, g_loc, offs = backend.regroup(cur["xr"][i], cur["gr"][i], kl, True, p.d)
            y_loc = backend.experts(p_loc, x_loc, offs, g_loc, r.w_gate, r.w_up, r.w_down,
                                    r.lora, st)
            y_src, _, _ = backend.regroup(y_loc, None, kl, False, p.d)
            y_back.append(y_src)
        ev_done = None
        if pipelined:
            ev_done = torch.cuda.Event()
            ev_done.record(main)
            for t in y_back:
                t.record_stream(side)
        # chunk c + 1's dispatch and transfer go on the side stream before chunk c's return
        # transfer, so they overlap chunk c's expert GEMMs
        if c + 1 < n:
            pending = dispatch_and_send(c + 1)
        with _on(side):
            if pipelined:
                side.wait_event(ev_done)
            # X3: results back to the ranks that own the tokens
            y_perm = xchg.all_to_all(y_back, cur["recv"], cur["send"])
            t0, t1 = bounds[c]
            for i, (r, st) in enumerate(zip(ranks, sts)):
                backend.combine(cur["pc"], y_perm[i], cur["chs"][i].slot_row, st.y[t0:t1], st)
    if pipelined:
        main.wait_stream(side)
    out = []
    counts_total = [cc.sum(dim=(0, 1)) for cc in cnt_all]
    partials_all = xchg.all_gather([st.partials for st in sts])
    p_total = moe.Problem(T=P * p.T, d=p.d, E=p.E, k=p.k, F=p.F, r=p.r,
                          lora_scale=p.lora_scale, cap_num=p.cap_num, cap_den=p.cap_den)
    for i, (r, st) in enumerate(zip(ranks, sts)):
        pa = partials_all[i].reshape(-1, p.E)
        aux = backend.aux(p_total, counts_total[i], pa, st)
        out.append(dict(y=st.y, aux=aux, plans=plans[i], state=st))
    return out
