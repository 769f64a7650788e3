"""Expert parallelism (EP) of the MoE layer across the GPUs of a node: each rank owns E / N of
the routed experts, and every token's rows travel to the ranks of its experts and back.

DeepSeek-V3 co-design teardown (wsisp.com) §2.3 gives the skeleton: the tokens sorted by
expert, the per-expert counts exchanged first, the rows exchanged by an all-to-all, the
experts run, and a reverse all-to-all brings the results back for the weighted sum.  The
Insights into DeepSeek-V3 précis §3.1 sends the dispatch in FP8 and the combine in BF16, with
the shared expert computed where the token lives.

One step on rank r (all kernels are libmoe's, the exchanges torch.distributed's all-to-all):
  1. gate, 1x128 quantisation and the permutation's indices, all local (routed experts only);
  2. the rows of each destination's experts, a contiguous range of the permutation, are
     gathered into the send buffer: FP8 codes [rows, H] and their FP32 scales [rows, H/128];
  3. the per-expert counts go to the owners (an all-to-all of E ints), which is what fixes
     every split of the row exchange (and forces the one host synchronisation of the step,
     as in the skeleton);
  4. the codes and scales are exchanged; the received rows arrive source-major with the
     experts of each source in order, and a one-slot permutation regroups them by local
     expert for the grouped GEMMs (gate/up with SwiGLU + requantisation, then down);
  5. the BF16 results go back to receive order and then, by the reverse all-to-all, to the
     ranks that sent the rows, in the order of their permutation;
  6. the shared expert runs on the rank's own tokens, and the combine forms the output.

The communication plan (splits, receive layout) is plain host logic kept apart from the
kernels, so that it can be exercised by gloo ranks on CPU tensors.
"""
import numpy as np
import torch
import torch.distributed as dist

from . import moe


def experts_per_rank(n_experts, world):
    if n_experts % world:
        raise ValueError("%d experts do not split evenly over %d ranks" % (n_experts, world))
    return n_experts // world


def send_splits(counts, world):
    """Rows for each destination: the rows of that rank's experts, which the permutation keeps
    contiguous and in rank order.  counts: the per-expert row counts (host ints, [E])."""
    c = np.asarray(counts, dtype=np.int64)
    ep = experts_per_rank(c.size, world)
    return [int(c[d * ep:(d + 1) * ep].sum()) for d in range(world)]


def exchange_counts(counts, world, group=None):
    """All-to-all of the per-expert row counts: rank d receives, from every source s, the counts
    of its own experts.  counts: int32 tensor [E] (device of the group's backend).  Returns the
    received counts [world, E / world] (same device)."""
    ep = experts_per_rank(counts.numel(), world)
    out = torch.empty_like(counts)
    if world == 1:
        out.copy_(counts)
    else:
        dist.all_to_all_single(out, counts.contiguous(), group=group)
    return out.view(world, ep)


def recv_expert_ids(recv_counts):
    """Local expert of every received row: the rows come source-major, and within a source in
    ascending expert order.  recv_counts: [world, E/world] host ints.  Returns int32 [rows]."""
    rc = np.asarray(recv_counts, dtype=np.int64)
    ep = rc.shape[1]
    return np.concatenate([np.repeat(np.arange(ep, dtype=np.int32), rc[s]) for s in range(rc.shape[0])]) \
        if rc.size else np.zeros(0, np.int32)


def exchange_rows(send, send_counts, recv_counts, group=None):
    """All-to-all of rows with variable splits: send [sum(send_counts), ...] -> the received
    rows [sum(recv_counts), ...] of the same trailing shape and dtype."""
    out = torch.empty((int(sum(recv_counts)),) + tuple(send.shape[1:]), dtype=send.dtype, device=send.device)
    if dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_to_all_single(out, send.contiguous(), output_split_sizes=list(recv_counts),
                               input_split_sizes=list(send_counts), group=group)
    else:
        out.copy_(send)
    return out


class EPLayer:
    """The MoE layer forward with the routed experts split over the ranks of `group` (one GPU
    each), in either FP8 mode.  weights: this rank's FP8 expert weights, its E / N routed experts followed by the
    shared expert (W13 [E/N + 1, 2I, H], W13_s, W2 [E/N + 1, H, I], W2_s, as moe_quant_128x128
    writes them) and the whole gate weight Wg [E, H] (BF16)."""

    def __init__(self, cfg, weights, group=None, device="cuda"):
        self.cfg = dict(cfg)
        if self.cfg["mode"] not in ("fp8", "mxfp8") or not self.cfg["has_shared"]:
            raise ValueError("the EP layer runs an FP8 mode with a shared expert")
        self.mx = self.cfg["mode"] == "mxfp8"  # power-of-two scales (weights from pow2=True)
        self.group = group
        self.world = dist.get_world_size(group) if dist.is_initialized() else 1
        self.rank = dist.get_rank(group) if dist.is_initialized() else 0
        self.E = cfg["n_experts"]
        self.ep = experts_per_rank(self.E, self.world)
        self.w = weights
        self.dev = device
        # the local permutation covers the routed experts only (the shared expert stays local)
        self.cfg_routed = dict(self.cfg, has_shared=0)
        # the receive-side regrouping: one slot per row over this rank's experts
        self.cfg_local = dict(self.cfg, n_experts=self.ep, n_group=1, topk_group=1, top_k=1, has_shared=0)
        if self.ep < 2:  # a one-expert group is outside moe_config's rules: regroup over two
            self.cfg_local.update(n_experts=2)

    def _slice(self, name, lo, hi):
        return self.w[name][lo:hi]

    def _down(self, n_groups, offs, rows, hq, hs, lo, hi, out):
        """The down-projection GEMM of experts [lo, hi) into BF16 rows."""
        c = self.cfg
        if self.mx:
            moe.moe_grouped_gemm_mxfp8(n_groups, offs, rows, c["hidden"], c["inter"], hq, hs, self._slice("W2", lo, hi),
                                       self._slice("W2_s", lo, hi), moe.MOE_EPI_STORE, out, None)
        else:
            moe.moe_grouped_gemm_fp8(n_groups, offs, rows, c["hidden"], c["inter"], hq, hs, self._slice("W2", lo, hi),
                                     self._slice("W2_s", lo, hi), moe.MOE_EPI_STORE, out, None, None)

    def forward(self, x, bias, y, topk_idx, topk_w, counts):
        c, H, I, K = self.cfg, self.cfg["hidden"], self.cfg["inter"], self.cfg["top_k"]
        T = x.shape[0]
        dev = self.dev
        u8, f32, i32 = torch.uint8, torch.float32, torch.int32
        # 1. local routing, quantisation, permutation indices
        moe.moe_gate(c, x, self.w["Wg"], bias, topk_idx, topk_w, counts)
        xq = torch.empty(T, H, dtype=u8, device=dev)
        xs = torch.empty(T, H // 128, dtype=f32, device=dev)
        (moe.moe_quant_1x128_pow2 if self.mx else moe.moe_quant_1x128)(x, xq, xs)
        R = T * K
        offs = torch.empty(self.E + 1, dtype=i32, device=dev)
        perm_tok = torch.empty(R, dtype=i32, device=dev)
        row_of = torch.empty(T, K, dtype=i32, device=dev)
        moe.moe_permute(self.cfg_routed, T, topk_idx, counts, xq, xs, offs, perm_tok, row_of, None, None,
                        moe.workspace(self.cfg_routed, T, dev))
        # 2. the send buffers, in the permutation's order
        send_q = torch.empty(R, H, dtype=u8, device=dev)
        send_s = torch.empty(R, H // 128, dtype=f32, device=dev)
        moe.moe_gather_rows(perm_tok, xq, send_q)
        moe.moe_gather_rows(perm_tok, xs, send_s)
        # 3. counts to the owners (the step's host synchronisation); the valid rows are the
        # first sum(counts) of the permutation, any rows of dropped slots come after them
        recv_counts = exchange_counts(counts, self.world, self.group).cpu().numpy()
        s_splits = send_splits(counts.cpu().numpy(), self.world)
        r_splits = [int(v) for v in recv_counts.sum(axis=1)]
        V = sum(s_splits)
        # 4. exchange, regroup by local expert, expert FFNs
        recv_q = exchange_rows(send_q[:V], s_splits, r_splits, self.group)
        recv_s = exchange_rows(send_s[:V], s_splits, r_splits, self.group)
        n = recv_q.shape[0]
        y_recv = torch.empty(n, H, dtype=torch.bfloat16, device=dev)
        if n > 0:
            ids = torch.from_numpy(recv_expert_ids(recv_counts)).to(dev).view(n, 1)
            El = self.cfg_local["n_experts"]
            offs_l = torch.empty(El + 1, dtype=i32, device=dev)
            perm_l = torch.empty(n, dtype=i32, device=dev)
            row_l = torch.empty(n, 1, dtype=i32, device=dev)
            cnt_l = torch.empty(El, dtype=i32, device=dev)
            moe.moe_permute(self.cfg_local, n, ids, cnt_l, recv_q, recv_s, offs_l, perm_l, row_l, None, None,
                            moe.workspace(self.cfg_local, n, dev))
            lo, hi = 0, self.ep
            hq = torch.empty(n, I, dtype=u8, device=dev)
            hs = torch.empty(I // 128, n, dtype=f32, device=dev)
            moe.moe_grouped_gemm_fp8_gather(self.ep, offs_l, n, 2 * I, H, perm_l, recv_q, recv_s,
                                            self._slice("W13", lo, hi), self._slice("W13_s", lo, hi),
                                            moe.MOE_EPI_SWIGLU_QUANT, hq, hs, mx=self.mx)
            yl = torch.empty(n, H, dtype=torch.bfloat16, device=dev)
            self._down(self.ep, offs_l, n, hq, hs, lo, hi, yl)
            # 5. back to receive order: a one-slot combine with weight 1 is an exact row gather
            ones = torch.ones(n, 1, dtype=f32, device=dev)
            moe.moe_combine(self.cfg_local, n, yl, row_l, ones, None, y_recv)
        y_routed = torch.empty(R, H, dtype=torch.bfloat16, device=dev)  # rows the combine may index
        y_routed[:V] = exchange_rows(y_recv, r_splits, s_splits, self.group)
        # 6. the shared expert on this rank's tokens, then the combine
        ident = torch.arange(T, dtype=i32, device=dev)
        offs_s = torch.tensor([0, T], dtype=i32, device=dev)
        hq_s = torch.empty(T, I, dtype=u8, device=dev)
        hs_s = torch.empty(I // 128, T, dtype=f32, device=dev)
        ysh = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        sh = self.ep
        moe.moe_grouped_gemm_fp8_gather(1, offs_s, T, 2 * I, H, ident, xq, xs, self._slice("W13", sh, sh + 1),
                                        self._slice("W13_s", sh, sh + 1), moe.MOE_EPI_SWIGLU_QUANT, hq_s, hs_s,
                                        mx=self.mx)
        self._down(1, offs_s, T, hq_s, hs_s, sh, sh + 1, ysh)
        moe.moe_combine(c, T, y_routed, row_of, topk_w, ysh, y)
        return dict(send=s_splits, recv=r_splits)
