"""A per-rank compute backend for the expert-parallel driver built from the fp64 oracle and
plain torch CPU ops (test infrastructure): it lets world_size-2 gloo tests run the EP
exchange logic on the CPU.  Each step computes what the matching C-ABI call computes
(moe_route, moe_expert_counts, moe_dispatch_ep, moe_ep_regroup, moe_expert_ffn,
moe_combine, moe_aux_loss), in float64."""

import numpy as np
import torch

import oracle


class OracleBackend:
    def __init__(self):
        self.dtype = torch.float64

    def route(self, p, x, w_router, bias, st):
        L = oracle.router_logits(x.numpy(), w_router.numpy(),
                                 None if bias is None else bias.numpy())
        idx, g, prob = oracle.route(L, p.k)
        st.topk_idx = torch.from_numpy(idx.astype(np.int64))
        st.topk_gate = torch.from_numpy(g)
        st.partials = torch.from_numpy(prob.sum(axis=0, keepdims=True))

    def counts(self, p, idx, st):
        return torch.bincount(idx.reshape(-1), minlength=p.E).to(torch.int64)

    def dispatch(self, p, C, idx, gate, x, pos_base, st):
        class Ch:
            pass
        ch = Ch()
        idx = idx.numpy()
        base = np.asarray(pos_base, dtype=np.int64)
        T, k = idx.shape
        queues = [[] for _ in range(p.E)]
        seen = np.zeros(p.E, dtype=np.int64)
        for t in range(T):
            for j in range(k):
                e = int(idx[t, j])
                pos = seen[e]
                seen[e] += 1
                if C is None or base[e] + pos < C:
                    queues[e].append(t * k + j)
        row_slot = np.array([s for q in queues for s in q], dtype=np.int64)
        offsets = np.zeros(p.E + 1, dtype=np.int64)
        offsets[1:] = np.cumsum([len(q) for q in queues])
        slot_row = np.full(T * k, -1, dtype=np.int64)
        slot_row[row_slot] = np.arange(len(row_slot))
        ch.offsets = torch.from_numpy(offsets)
        ch.slot_row = torch.from_numpy(slot_row)
        ch.row_slot = torch.from_numpy(row_slot)
        ch.x_perm = x[torch.from_numpy(row_slot // k)].to(self.dtype)
        ch.gate_perm = gate.reshape(-1)[torch.from_numpy(row_slot)]
        return ch

    def regroup(self, src, gsrc, kept, to_expert, d):
        P, El = kept.shape
        se = [(s, e) for s in range(P) for e in range(El)]
        es = [(s, e) for e in range(El) for s in range(P)]
        start = {}
        order_from, order_to = (se, es) if to_expert else (es, se)
        off = 0
        for s, e in order_from:
            start[(s, e)] = off
            off += int(kept[s, e])
        idx = []
        for s, e in order_to:
            idx.extend(range(start[(s, e)], start[(s, e)] + int(kept[s, e])))
        idx = torch.tensor(idx, dtype=torch.int64)
        dst = src[idx]
        gdst = None if gsrc is None else gsrc[idx]
        offs = None
        if to_expert:
            per = kept.sum(axis=0)
            offs = torch.from_numpy(np.concatenate([[0], np.cumsum(per)]).astype(np.int64))
        return dst, gdst, offs

    def experts(self, p_loc, x_loc, offsets, gates, w_gate, w_up, w_down, lora, st):
        y = torch.zeros((x_loc.shape[0], p_loc.d), dtype=self.dtype)
        for e in range(p_loc.E):
            lo, hi = int(offsets[e]), int(offsets[e + 1])
            if hi == lo:
                continue
            L = None if lora is None else {n: v[e].numpy() for n, v in lora.items()}
            o = oracle.expert_forward(x_loc[lo:hi].numpy(), w_gate[e].numpy(), w_up[e].numpy(),
                                      w_down[e].numpy(), L, p_loc.lora_scale)[3]
            y[lo:hi] = gates[lo:hi, None] * torch.from_numpy(o)
        return y

    def combine(self, p, y_perm, slot_row, y_out, st):
        sr = slot_row.numpy()
        y_out.zero_()
        for t in range(p.T):
            for j in range(p.k):
                r = sr[t * p.k + j]
                if r >= 0:
                    y_out[t] += y_perm[r]

    def new_output(self, T, d):
        return torch.zeros((T, d), dtype=self.dtype)

    def aux(self, p_total, counts_total, partials_all, st):
        f = counts_total.to(torch.float64) / (p_total.T * p_total.k)
        P = partials_all.sum(dim=0) / p_total.T
        return torch.tensor([float(p_total.E * (f * P).sum())], dtype=torch.float64)
