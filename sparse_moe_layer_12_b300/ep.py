"""Expert-parallel MoE layer: routed experts split over ranks, all-to-all dispatch and combine.

"DeepSeek-V3 Overview and Key Innovations" (Training Infrastructure and Optimization):
the experts are spread over GPUs and tokens travel to them and back with all-to-all
dispatch / combine kernels over NVLink and InfiniBand; "拆解DeepSeek V3" gives the node
(8 GPUs over NVLink / NVSwitch); "DeepSeek-V3 详解" 2.4: node-limited routing keeps a
token's experts on few nodes (moe_route's group-limited routing, with one group per rank
or node).

Layout: the E routed experts form G contiguous ranges of E_loc = E / G; rank r owns
experts [r E_loc, (r + 1) E_loc).  The router and the shared experts are replicated, and
every rank routes its own T tokens.  One layer step on rank r:

  1. moe_route and moe_permute: the expert-major copy of x is already ordered by
     destination rank, rows for rank r' are one contiguous range;
  2. all-to-all of the per-expert counts -> recv_counts [G, E_loc]; the row split sizes
     go to the host (one small device-to-host copy: the collective needs them there);
  3. all-to-all of the permuted rows (and, on the FP8 path, their 1x128 scales): rows
     arrive source-major;
  4. moe_ep_regroup to local expert-major order, moe_expert_ffn over the E_loc local
     experts, moe_ep_regroup back to source-major order;
  5. all-to-all of the expert outputs with the inverse splits: they land in this rank's
     permuted order, rows 0 .. T k - 1 of y;
  6. the shared experts on the rank's own tokens (one-expert moe_expert_ffn calls) into
     rows T k + s T .. of y;
  7. moe_combine, and the bias update from the all-reduced counts with the global token
     count (every rank applies the same update, as the data-parallel replicas do).

The compute calls come from an `ops` object (CudaOps: the C-ABI library); the exchanges
from a `transport` (DistTransport: torch.distributed, NCCL on GPUs; LocalTransport:
ranks emulated as threads of one process, exchanges as device copies -- no kernel of one
rank waits on another's).
"""
from __future__ import annotations

import threading

import torch


# ---------------------------------------------------------------- transports


class DistTransport:
    """Exchanges through torch.distributed (NCCL between GPUs, gloo on CPUs)."""

    def __init__(self, group=None):
        import torch.distributed as dist

        self.dist, self.group = dist, group

    def all_to_all(self, out, inp, out_splits=None, in_splits=None):
        self.dist.all_to_all_single(out, inp, out_splits, in_splits, group=self.group)

    def all_reduce_sum(self, t):
        self.dist.all_reduce(t, op=self.dist.ReduceOp.SUM, group=self.group)


class LocalTransport:
    """G ranks as threads of one process; every exchange is a set of tensor copies made
    after all ranks have posted their inputs (a barrier on each side)."""

    def __init__(self, world: int):
        self.world = world
        self._barrier = threading.Barrier(world)
        self._posted = [None] * world

    def view(self, rank: int) -> "_LocalRank":
        return _LocalRank(self, rank)


class _LocalRank:
    def __init__(self, hub: LocalTransport, rank: int):
        self.hub, self.rank = hub, rank

    def all_to_all(self, out, inp, out_splits=None, in_splits=None):
        G = self.hub.world
        in_splits = in_splits or [inp.shape[0] // G] * G
        out_splits = out_splits or [out.shape[0] // G] * G
        self.hub._posted[self.rank] = (inp, list(in_splits))
        self.hub._barrier.wait()
        o = 0
        for src in range(G):
            t, splits = self.hub._posted[src]
            lo = sum(splits[: self.rank])
            n = splits[self.rank]
            if n != out_splits[src]:
                raise RuntimeError(f"rank {self.rank}: {n} rows from rank {src}, expected {out_splits[src]}")
            if n:
                out[o:o + n].copy_(t[lo:lo + n])
            o += n
        self.hub._barrier.wait()

    def all_reduce_sum(self, t):
        self.hub._posted[self.rank] = (t.clone(), None)
        self.hub._barrier.wait()
        acc = self.hub._posted[0][0].clone()
        for src in range(1, self.hub.world):
            acc += self.hub._posted[src][0]
        self.hub._barrier.wait()
        t.copy_(acc)


# ---------------------------------------------------------------- one rank


def expert_range(E: int, world: int, rank: int) -> tuple[int, int]:
    """Routed experts [lo, hi) owned by `rank`."""
    if E % world:
        raise ValueError(f"E = {E} experts do not split evenly over {world} ranks")
    n = E // world
    return rank * n, (rank + 1) * n


class EPRank:
    """The per-rank part of the expert-parallel layer (steps 1-7 above)."""

    def __init__(self, ops, transport, T: int, d: int, E: int, S: int, k: int, rank: int, world: int):
        if E % world:
            raise ValueError(f"E = {E} experts do not split evenly over {world} ranks")
        self.ops, self.tp = ops, transport
        self.T, self.d, self.E, self.S, self.k = T, d, E, S, k
        self.rank, self.world, self.E_loc = rank, world, E // world

    def forward(self, x, bias, logit_offset=None, update_bias=False, gamma=0.001):
        """Returns (out [T, d], topk_idx, topk_gate, counts of this rank's tokens)."""
        ops, tp, G, E_loc = self.ops, self.tp, self.world, self.E_loc
        T, d, S, k = self.T, self.d, self.S, self.k
        idx, gate, counts, offsets = ops.route(x, bias, logit_offset)
        xp, xps, inv = ops.permute(x, idx, offsets)
        send_counts = counts.view(G, E_loc)
        recv_counts = torch.empty_like(send_counts)
        tp.all_to_all(recv_counts, send_counts)
        sizes = torch.cat([send_counts.sum(1), recv_counts.sum(1)]).cpu().tolist()
        send_splits, recv_splits = sizes[:G], sizes[G:]
        R = sum(recv_splits)
        x_recv = torch.empty((R,) + tuple(xp.shape[1:]), dtype=xp.dtype, device=xp.device)
        tp.all_to_all(_wire(x_recv), _wire(xp), recv_splits, send_splits)
        xs_recv = None
        if xps is not None:
            xs_recv = torch.empty((R, xps.shape[1]), dtype=xps.dtype, device=xps.device)
            tp.all_to_all(xs_recv, xps, recv_splits, send_splits)
        x_loc, xs_loc, loc_off = ops.regroup(recv_counts, x_recv, xs_recv, True)
        y_loc = ops.local_ffn(x_loc, xs_loc, loc_off)
        y_ret, _, _ = ops.regroup(recv_counts, y_loc, None, False)
        y = torch.empty((T * k + S * T, d), dtype=y_loc.dtype, device=y_loc.device)
        tp.all_to_all(_wire(y[: T * k]), _wire(y_ret), send_splits, recv_splits)
        for s in range(S):
            ops.shared_ffn(x, s, y[T * k + s * T: T * k + (s + 1) * T])
        out = ops.combine(y, gate, inv)
        if update_bias:
            c = counts.clone()
            tp.all_reduce_sum(c)
            t = torch.tensor([T], dtype=torch.int64, device=c.device)
            tp.all_reduce_sum(t)
            ops.bias_update(c, bias, int(t.item()), gamma)
        return out, idx, gate, counts


def _wire(t):
    """The bytes a collective moves: float8 rows travel as uint8."""
    return t.view(torch.uint8) if t.dtype == torch.float8_e4m3fn else t


# ---------------------------------------------------------------- the CUDA library as ops


class CudaOps:
    """The C-ABI calls of one rank: the full router (replicated), this rank's E_loc routed
    experts and the shared experts.  Weights: w_gate_up_local [E_loc, 2I, d] and
    w_down_local [E_loc, d, I] (bf16, or E4M3 with 128x128 block scales), shared experts
    w_gate_up_shared [S, 2I, d] / w_down_shared [S, d, I] likewise."""

    def __init__(self, T, d, E, S, k, I, world, w_router, w_gate_up_local, w_down_local, w_gate_up_shared,
                 w_down_shared, fp8=False, scales=None, n_group=0, topk_group=0, pow2=False):
        from sparse_moe_layer_12_b300 import binding as B

        self.B = B
        self.T, self.d, self.E, self.S, self.k, self.I, self.fp8, self.pow2 = T, d, E, S, k, I, fp8, pow2
        self.E_loc = E // world
        self.wr = w_router
        self.wgu, self.wd = w_gate_up_local, w_down_local
        self.wgu_sh, self.wd_sh = w_gate_up_shared, w_down_shared
        sc = scales or {}
        self.gs, self.ds = sc.get("gate_up_local"), sc.get("down_local")
        self.gs_sh, self.ds_sh = sc.get("gate_up_shared"), sc.get("down_shared")
        self.shape = B.make_shape(T, d, E, S, k, I, fp8, n_group, topk_group, pow2=pow2)
        # one shared expert as a dense one-expert layer
        self.shape_sh = B.make_shape(T, d, 1, 0, 1, I, fp8, pow2=pow2)
        self.ws = B.alloc_workspace(self.shape, w_router.device)
        self.ws_sh = B.alloc_workspace(self.shape_sh, w_router.device)
        self._ws_loc = None
        self.sh_off = torch.tensor([0, T], dtype=torch.int32, device=w_router.device)
        self.sh_idx = torch.zeros(T, 1, dtype=torch.int32, device=w_router.device)

    def route(self, x, bias, logit_offset):
        return self.B.moe_route(self.shape, x, self.wr, bias, logit_offset, ws=self.ws)

    def permute(self, x, idx, offsets):
        xp, xps, _, inv = self.B.moe_permute(self.shape, x, idx, offsets, ws=self.ws)
        return xp, xps, inv

    def regroup(self, recv_counts, src, src_scale, to_local):
        return self.B.moe_ep_regroup(recv_counts, src, to_local, self.ws, src_scale=src_scale)

    def local_ffn(self, x_loc, xs_loc, loc_off):
        R = x_loc.shape[0]
        B = self.B
        shape = B.make_shape(R, self.d, self.E_loc, 0, 1, self.I, self.fp8, pow2=self.pow2)
        need = B.workspace_bytes(shape)
        if self._ws_loc is None or self._ws_loc.numel() < need:
            self._ws_loc = B.alloc_workspace(shape, x_loc.device)
        # the bf16 rows of the shared experts: none here (S = 0), any buffer of the shape will do
        x_in = x_loc if not self.fp8 else torch.empty(R, self.d, dtype=torch.bfloat16, device=x_loc.device)
        return B.moe_expert_ffn(shape, x_loc, xs_loc, x_in, loc_off, self.wgu, self.wd, self.gs, self.ds,
                                ws=self._ws_loc)

    def shared_ffn(self, x, s, y_out):
        B = self.B
        if self.fp8:  # the shared expert's input rows quantised per 1x128, as moe_permute does
            xq, xqs, _, _ = B.moe_permute(self.shape_sh, x, self.sh_idx, self.sh_off, ws=self.ws_sh)
        else:
            xq, xqs = x, None
        B.moe_expert_ffn(self.shape_sh, xq, xqs, x, self.sh_off, self.wgu_sh[s:s + 1], self.wd_sh[s:s + 1],
                         None if self.gs_sh is None else self.gs_sh[s:s + 1],
                         None if self.ds_sh is None else self.ds_sh[s:s + 1], ws=self.ws_sh, y=y_out)

    def combine(self, y, gate, inv):
        return self.B.moe_combine(self.shape, y, gate, inv)

    def bias_update(self, counts, bias, T_global, gamma):
        B = self.B
        B.moe_bias_update(B.make_shape(T_global, self.d, self.E, self.S, self.k, self.I, self.fp8, pow2=self.pow2),
                          counts, bias, gamma)

    def device_status(self) -> int:
        """The first non-OK device status of this rank's workspaces (read and cleared)."""
        for ws in (self.ws, self.ws_sh, self._ws_loc):
            if ws is not None:
                st = self.B.moe_get_device_status(ws)
                if st:
                    return st
        return 0
