"""The replica path with two gloo ranks on CPU: each rank greedily decodes its
share of the prompts with the CPU oracle standing in for a GPU replica; the
gathered tokens equal a single-process run and the job time is the slowest
rank's."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from invariant_fixed_order_gb300 import replicas


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def tiny_model():
    rng = np.random.default_rng(3)
    d, H, Hkv, Dh, F, V = 64, 4, 2, 16, 128, 96

    def w(*shape, std=0.05, mean=0.0):
        import torch
        return torch.from_numpy(rng.standard_normal(shape) * std + mean).float().to(torch.bfloat16).float().numpy()

    layer = {"gamma_attn": w(d, mean=1.0, std=0.02), "w_qkv": w((H + 2 * Hkv) * Dh, d), "w_o": w(d, H * Dh),
             "gamma_ffn": w(d, mean=1.0, std=0.02), "w_gate": w(F, d), "w_up": w(F, d), "w_down": w(d, F)}
    head = {"embed": w(V, d, std=1.0), "gamma_final": w(d, mean=1.0, std=0.02), "w_lm": w(V, d)}
    return (d, H, Hkv, Dh, F, V), layer, head


def greedy(prompt, n_new):
    import oracle
    (d, H, Hkv, Dh, F, V), layer, head = tiny_model()
    dims = oracle.Dims(d, H, Hkv, Dh, F)
    toks = list(prompt)
    for _ in range(n_new):
        x = oracle.embed(head["embed"], toks)
        empty = [np.zeros((1, Hkv, Dh), np.float32)]
        xo, _, _, _ = oracle.layer_forward(dims, layer, [len(toks)], [0], empty, empty, x)
        _, t = oracle.lm_head(dims, head["gamma_final"], head["w_lm"], xo, [len(toks) - 1])
        toks.append(int(t[0]))
    return toks[len(prompt):]


PROMPTS = [[int(t) for t in np.random.default_rng(10 + i).integers(0, 96, 3 + 2 * i)] for i in range(5)]


def rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = replicas.shard(len(PROMPTS), world, rank)
    local = {i: greedy(PROMPTS[i], 3) for i in mine}
    allres = replicas.gather(local)
    slowest = replicas.max_over_ranks(10.0 + rank)
    q.put((rank, mine, allres, slowest))
    dist.barrier()
    dist.destroy_process_group()


def test_shard_partitions_every_item_once():
    for n in (0, 1, 5, 64):
        for world in (1, 2, 3, 8):
            got = sorted(i for r in range(world) for i in replicas.shard(n, world, r))
            assert got == list(range(n))
    with pytest.raises(ValueError):
        replicas.shard(4, 2, 2)


def test_two_gloo_replicas_match_one_process():
    import oracle
    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=300) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    single = {i: greedy(p, 3) for i, p in enumerate(PROMPTS)}
    shares = {r: mine for r, mine, _, _ in out}
    assert sorted(shares[0] + shares[1]) == list(range(len(PROMPTS)))
    for r, mine, allres, slowest in out:
        assert allres == single
        assert slowest == 11.0
