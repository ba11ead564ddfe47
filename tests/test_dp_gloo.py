"""The multi-GPU host logic (token shards, all-reduce of the per-expert load, bias
update with the global token count) on world_size-2 gloo ranks on CPU: the replicas'
biases must equal the single-process update over all tokens, bit for bit."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import moe_oracle as O
from sparse_moe_layer_12_b300 import dp
from sparse_moe_layer_12_b300 import inputs as I


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_update(counts, bias, T_global, gamma, k):
    new = O.bias_update(bias.numpy(), counts.numpy(), T_global, k, gamma)
    bias.copy_(torch.from_numpy(new))


def _worker(rank, world, port, T_global, steps, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    cfg = I.CONFIGS["tiny"].with_(T=T_global)
    x = I.make_x(cfg)
    wr = I.make_router(cfg)
    lo, hi = dp.shard_rows(T_global, rank, world)
    bias = torch.zeros(cfg.E)
    assert dp.global_token_count(hi - lo) == T_global
    for _ in range(steps):
        r = O.route(x[lo:hi].float().numpy(), wr.float().numpy(), bias.numpy(), cfg.k)
        counts = torch.from_numpy(O.expert_counts(r["idx"], cfg.E).astype(np.int32))
        dp.bias_update_global(counts, bias, T_global, cfg.gamma,
                              lambda c, b, T, g: _oracle_update(c, b, T, g, cfg.k))
    np.save(os.path.join(out_dir, f"bias{rank}.npy"), bias.numpy())
    dist.destroy_process_group()


def test_shards_cover_tokens():
    for T in (1, 7, 256, 1001):
        for world in (1, 2, 3, 8):
            spans = [dp.shard_rows(T, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == T
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            assert max(h - l for l, h in spans) - min(h - l for l, h in spans) <= 1


def test_replicas_keep_identical_bias(tmp_path):
    T_global, steps, world = 301, 5, 2
    mp.spawn(_worker, args=(world, _free_port(), T_global, steps, str(tmp_path)), nprocs=world, join=True)
    b0 = np.load(tmp_path / "bias0.npy")
    b1 = np.load(tmp_path / "bias1.npy")
    np.testing.assert_array_equal(b0, b1)
    # single process over all tokens
    cfg = I.CONFIGS["tiny"].with_(T=T_global)
    x = I.make_x(cfg).float().numpy()
    wr = I.make_router(cfg).float().numpy()
    b = np.zeros(cfg.E, np.float32)
    for _ in range(steps):
        r = O.route(x, wr, b, cfg.k)
        b = O.bias_update(b, O.expert_counts(r["idx"], cfg.E), T_global, cfg.k, cfg.gamma)
    np.testing.assert_array_equal(b0, b)
    assert np.any(b != 0)
