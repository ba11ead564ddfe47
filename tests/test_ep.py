"""The expert-parallel host logic (sparse_moe_layer_12_b300/ep.py) on the CPU: split
sizes, the three all-to-all exchanges, the regroup directions, where the returned rows
and the shared experts land in y, and the bias update from the global load.

The compute calls are the oracle's (float64), the regroup a stable sort of the received
rows by local expert; ranks run as threads (LocalTransport, 2 and 4 ranks) and as gloo
processes (2 ranks).  Each rank's output must equal the oracle layer over all E experts
on that rank's tokens, and every rank's bias the single update from the summed loads."""
import os
import socket
import threading

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import moe_oracle as O
from sparse_moe_layer_12_b300 import ep


class OracleOps:
    """The layer's calls for one rank in float64 on the CPU, from the oracle."""

    def __init__(self, T, d, E, S, k, world, rank, wr, wgu, wd):
        self.T, self.d, self.E, self.S, self.k = T, d, E, S, k
        lo, hi = ep.expert_range(E, world, rank)
        self.E_loc = hi - lo
        self.wr = wr
        self.wgu_loc, self.wd_loc = wgu[lo:hi], wd[lo:hi]
        self.wgu_sh, self.wd_sh = wgu[E:E + S], wd[E:E + S]

    def route(self, x, bias, logit_offset):
        r = O.route(x.numpy(), self.wr, bias.numpy(), self.k, None if logit_offset is None else logit_offset.numpy())
        counts = O.expert_counts(r["idx"], self.E)
        return (torch.from_numpy(r["idx"]), torch.from_numpy(r["gate"]), torch.from_numpy(counts),
                torch.from_numpy(O.offsets_from_counts(counts)))

    def permute(self, x, idx, offsets):
        p = O.permutation(idx.numpy(), self.E)
        return x[torch.from_numpy(p["perm_token"]).long()], None, torch.from_numpy(p["inv_pos"])

    def regroup(self, recv_counts, src, src_scale, to_local):
        c = recv_counts.numpy()
        G, E_loc = c.shape
        # received rows are source-major, expert-major inside a source: a stable sort by
        # local expert puts them expert-major with the sources in order
        expert_of_row = np.concatenate([np.repeat(np.arange(E_loc), c[s]) for s in range(G)])
        order = torch.from_numpy(np.argsort(expert_of_row, kind="stable"))
        if to_local:
            dst = src[order]
        else:
            dst = torch.empty_like(src)
            dst[order] = src
        off = torch.from_numpy(O.offsets_from_counts(c.sum(0)))
        return dst, None, off

    def local_ffn(self, x_loc, xs_loc, loc_off):
        y = torch.zeros(x_loc.shape[0], self.d, dtype=torch.float64)
        for e in range(self.E_loc):
            lo, hi = int(loc_off[e]), int(loc_off[e + 1])
            if hi > lo:
                y[lo:hi] = torch.from_numpy(O.swiglu_expert(x_loc[lo:hi].numpy(), self.wgu_loc[e], self.wd_loc[e]))
        return y

    def shared_ffn(self, x, s, y_out):
        y_out.copy_(torch.from_numpy(O.swiglu_expert(x.numpy(), self.wgu_sh[s], self.wd_sh[s])))

    def combine(self, y, gate, inv):
        return torch.from_numpy(O.combine(y.numpy(), gate.numpy(), inv.numpy(), self.T, self.k, self.S))

    def bias_update(self, counts, bias, T_global, gamma):
        bias.copy_(torch.from_numpy(O.bias_update(bias.numpy(), counts.numpy(), T_global, self.k, gamma)))


def _layer(T=37, d=16, E=8, S=2, k=3, I=8, world=2, seed=0):
    rng = np.random.default_rng(seed)
    wr = rng.standard_normal((E, d)) * 0.5
    wgu = rng.standard_normal((E + S, 2 * I, d)) / np.sqrt(d)
    wd = rng.standard_normal((E + S, d, I)) / np.sqrt(I)
    xs = [torch.from_numpy(rng.standard_normal((T, d))) for _ in range(world)]
    bias = rng.uniform(-0.05, 0.05, E).astype(np.float32)
    return dict(T=T, d=d, E=E, S=S, k=k, I=I, world=world, wr=wr, wgu=wgu, wd=wd, xs=xs, bias=bias)


def _expected(L):
    outs, counts = [], np.zeros(L["E"], dtype=np.int64)
    for x in L["xs"]:
        res = O.forward(x.numpy(), L["wr"], L["bias"], L["wgu"], L["wd"], L["k"], L["S"])
        outs.append(res["out"])
        counts += O.expert_counts(res["route"]["idx"], L["E"])
    b = O.bias_update(L["bias"], counts, L["T"] * L["world"], L["k"], 0.001)
    return outs, b


def _rank_forward(L, rank, transport):
    ops = OracleOps(L["T"], L["d"], L["E"], L["S"], L["k"], L["world"], rank, L["wr"], L["wgu"], L["wd"])
    r = ep.EPRank(ops, transport, L["T"], L["d"], L["E"], L["S"], L["k"], rank, L["world"])
    bias = torch.from_numpy(L["bias"].copy())
    out, *_ = r.forward(L["xs"][rank], bias, update_bias=True, gamma=0.001)
    return out.numpy(), bias.numpy()


@pytest.mark.parametrize("world,E,S", [(2, 8, 2), (4, 8, 1), (4, 16, 0)])
def test_ep_threads_match_the_layer(world, E, S):
    L = _layer(E=E, S=S, world=world, seed=world + E)
    want, want_b = _expected(L)
    hub = ep.LocalTransport(world)
    res, errs = [None] * world, []

    def run(rank):
        try:
            res[rank] = _rank_forward(L, rank, hub.view(rank))
        except Exception as exc:  # surfaced below
            errs.append(exc)
            hub._barrier.abort()

    th = [threading.Thread(target=run, args=(r,)) for r in range(world)]
    for t in th:
        t.start()
    for t in th:
        t.join(60)
    assert not errs, errs
    for rank in range(world):
        out, b = res[rank]
        np.testing.assert_allclose(out, want[rank], rtol=1e-12, atol=1e-12)
        np.testing.assert_array_equal(b, want_b)


def test_ep_rank_with_no_rows_for_a_rank():
    # every token picks experts of rank 0 only: rank 1 receives nothing and sends back nothing
    L = _layer(E=4, S=1, k=2, world=2, seed=9)
    L["wr"][2:] = 0.0
    L["wr"][:2] = np.abs(L["wr"][:2]) * 0 + 1.0
    L["xs"] = [x.abs() + 0.1 for x in L["xs"]]  # positive logits for experts 0 and 1, zero for 2 and 3
    want, want_b = _expected(L)
    hub = ep.LocalTransport(2)
    res = [None, None]
    th = [threading.Thread(target=lambda r=r: res.__setitem__(r, _rank_forward(L, r, hub.view(r)))) for r in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join(60)
    for rank in range(2):
        np.testing.assert_allclose(res[rank][0], want[rank], rtol=1e-12, atol=1e-12)
        np.testing.assert_array_equal(res[rank][1], want_b)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _gloo_worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        L = _layer(world=world, seed=3)
        out, b = _rank_forward(L, rank, ep.DistTransport())
        np.save(os.path.join(out_dir, f"out{rank}.npy"), out)
        np.save(os.path.join(out_dir, f"bias{rank}.npy"), b)
    finally:
        dist.destroy_process_group()


def test_ep_gloo_two_ranks(tmp_path):
    world = 2
    mp.spawn(_gloo_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world)
    L = _layer(world=world, seed=3)
    want, want_b = _expected(L)
    for rank in range(world):
        np.testing.assert_allclose(np.load(tmp_path / f"out{rank}.npy"), want[rank], rtol=1e-12, atol=1e-12)
        np.testing.assert_array_equal(np.load(tmp_path / f"bias{rank}.npy"), want_b)


def test_expert_range():
    assert ep.expert_range(256, 8, 3) == (96, 128)
    with pytest.raises(ValueError):
        ep.expert_range(10, 4, 0)
