"""KDA context parallelism (KCP) over the token axis.

"Kimi K3: KDA, attention residuals and Stable LatentMoE", Sec. 10.2: the KDA
recurrence is not additive, so a segment's effect on the state depends on the
state it starts from.  With M_t = (I - beta_t k_t k_t^T) Diag(alpha_t), a segment
acts as S_exit = M S_entry + S~, M = M_T ... M_1 and S~ its state from zero.
Each rank computes (M, S~) for its segment, one all-gather exchanges the pairs
(fixed size: a d_k x d_k and a d_k x d_v matrix per head), and rank i recovers
its entry state by applying the earlier ranks' pairs in order,
S <- M_j S + S~_j, before running its own segment from that state.

The per-rank steps are supplied by an operations object, so the same host
logic drives this library's kernels (`GpuOps`) or any other implementation of
the three steps:

    pair(seg)          -> (M [H, dk, dk], S~ [H, dk, dv])
    apply(M, S, St)    -> M S + St   (per head)
    prefill(seg, S0)   -> (o, S_T [H, dk, dv], y) of the segment from S0 [H, dk, dv]

A segment `seg` is a dict of one sequence's tokens on this rank: q, k, v, z,
beta, A, and optionally g_in, norm_w.
"""
from __future__ import annotations

import torch


class GpuOps:
    """The per-rank KCP steps on this library's kernels (device tensors).

    A segment's three state passes (M from S0 = I with v = 0, S~ from zero,
    its outputs from the entry state) share one set of chunk records: with
    bf16 q/k/v and d = 128 the records are built once (``kda_prefill_records``)
    and each pass is a ``kda_prefill_scan`` over them, M with the zero-v flag.
    Other inputs take three ``kda_prefill`` calls.
    """

    REC_KW = ("g_min", "qk_l2norm", "gate")
    SCAN_KW = ("scale", "norm_eps")

    def __init__(self, reuse_records=True, **prefill_kw):
        self.kw = dict(workspace="cache")
        self.kw.update(prefill_kw)
        self.reuse = reuse_records
        self._rec = {}   # id(seg) -> (seg, Records)

    def _records(self, seg):
        from . import kda
        k = seg["k"]
        if not (self.reuse and k.dtype == torch.bfloat16 and k.shape[2] == 128 and seg["v"].shape[2] == 128):
            return None
        hit = self._rec.get(id(seg))
        if hit is not None and hit[0] is seg:
            return hit[1]
        rec = kda.prefill_records(seg["q"], k, seg["v"], seg["z"], seg["beta"], seg["A"],
                                  **{n: self.kw[n] for n in self.REC_KW if n in self.kw})
        self._rec[id(seg)] = (seg, rec)
        return rec

    def _scan_kw(self):
        return {n: self.kw[n] for n in self.SCAN_KW if n in self.kw}

    def pair(self, seg):
        from . import kda
        k = seg["k"]
        H, dk = k.shape[1], k.shape[2]
        eye = torch.eye(dk, dtype=torch.float32, device=k.device).expand(1, H, dk, dk).contiguous()
        rec = self._records(seg)
        if rec is not None:
            _, M, _ = kda.prefill_scan(rec, S0=eye, want_o=False, zero_v=True, **self._scan_kw())
            _, St, _ = kda.prefill_scan(rec, want_o=False, **self._scan_kw())
            return M[0], St[0]
        # M: the state after the segment from S0 = I with v = 0 (dv = dk)
        _, M, _ = kda.prefill(seg["q"], k, torch.zeros_like(seg["v"]), seg["z"], seg["beta"], seg["A"],
                              S0=eye, want_o=False, **self.kw)
        # S~: the state after the segment from zero
        _, St, _ = kda.prefill(seg["q"], k, seg["v"], seg["z"], seg["beta"], seg["A"], want_o=False, **self.kw)
        return M[0], St[0]

    def apply(self, M, S, St):
        from . import kda
        X = S.contiguous().clone()
        return kda.kcp_apply(M.contiguous(), X, St.contiguous())

    def prefill(self, seg, S0):
        from . import kda
        rec = self._records(seg)
        if rec is not None:
            o, S_T, y = kda.prefill_scan(rec, S0=S0.unsqueeze(0).contiguous(), g_in=seg.get("g_in"),
                                         norm_w=seg.get("norm_w"), **self._scan_kw())
            self._rec.pop(id(seg), None)   # the segment's last pass
            return o, S_T[0], y
        o, S_T, y = kda.prefill(seg["q"], seg["k"], seg["v"], seg["z"], seg["beta"], seg["A"],
                                S0=S0.unsqueeze(0).contiguous(), g_in=seg.get("g_in"), norm_w=seg.get("norm_w"),
                                **self.kw)
        return o, S_T[0], y


def entry_state(pairs, S_init, ops):
    """Apply segments' pairs in order to S_init: S <- M_j S + S~_j."""
    S = S_init
    for M, St in pairs:
        S = ops.apply(M, S, St)
    return S


def kcp_prefill(seg, ops, group=None, S_init=None):
    """This rank's part of a KCP prefill of one sequence whose consecutive
    segments are held by the ranks of `group` in rank order.

    Returns (o, S_T, y) of the local segment; the last rank's S_T is the
    sequence's final state.  S_init: the state before the first segment
    ([H, dk, dv], None = zero), passed identically on every rank.
    """
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    M, St = ops.pair(seg)
    payload = torch.cat([M, St], dim=-1).contiguous()          # [H, dk, dk + dv]
    gathered = [torch.empty_like(payload) for _ in range(world)]
    dist.all_gather(gathered, payload, group=group)
    dk = M.shape[-1]
    S0 = torch.zeros_like(St) if S_init is None else S_init.to(St)
    pairs = [(g[..., :dk], g[..., dk:]) for g in gathered[:rank]]
    return ops.prefill(seg, entry_state(pairs, S0, ops))


def kcp_prefill_local(segments, ops, S_init=None):
    """The same algebra on one device: every segment's pair, then each segment
    from the entry state its predecessors give (a rank's view, in turn).
    Returns the list of per-segment (o, S_T, y)."""
    pairs = [ops.pair(seg) for seg in segments]
    St0 = pairs[0][1]
    S = torch.zeros_like(St0) if S_init is None else S_init.to(St0)
    out = []
    for i, seg in enumerate(segments):
        out.append(ops.prefill(seg, S))
        S = ops.apply(pairs[i][0], S, pairs[i][1])
    return out
