"""CUDA-graph replay with bucket padding as a fuzz axis ("Batch invariance and
reproducible inference", "The regression that only reproduces at one batch
size"): for random decode batches, a request's logits are the same bits from
an eager step, from the replay of the smallest bucket that holds the batch
(padded) and from the replay of a larger bucket."""
import numpy as np
import pytest
import torch

from invariant_fixed_order_gb300 import synth
from invariant_fixed_order_gb300.config import LLAMA3_8B_1L, TINY

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from invariant_fixed_order_gb300 import bi
    from invariant_fixed_order_gb300.engine import Engine
    from invariant_fixed_order_gb300.graphs import DecodeGraphs
    return bi, Engine, DecodeGraphs


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int32).cpu().numpy()


def run_fuzz(bi, Engine, DecodeGraphs, cfg, n_req, lo, hi, n_iter, ladder, seed):
    rng = np.random.default_rng(seed)
    max_ctx = hi + n_iter + 2
    max_pages = (max_ctx + 15) // 16
    n_max = max(ladder)
    eng = Engine(cfg, num_pages=n_req * max_pages + 8, max_pages=max_pages, max_T=max(hi, n_max), max_B=n_max,
                 max_R=max(hi, n_max))
    lens = rng.integers(lo, hi + 1, n_req)
    tables = np.zeros((n_req, max_pages), np.int32)
    last_tok, ctx = np.zeros(n_req, np.int32), np.zeros(n_req, np.int32)
    for i, n in enumerate(lens):
        tables[i] = eng.pool.alloc(max_pages)
        ids = synth.token_ids(int(n), cfg.V, seed * 100 + i)
        _, tok, _ = eng.step([int(n)], [0], ids, tables[i:i + 1], [int(n) - 1])
        last_tok[i], ctx[i] = int(tok[0].item()), int(n)
    graphs = DecodeGraphs(eng, max_ctx, ladder=ladder)
    buckets = sorted(graphs.buckets)
    checked = 0
    for it in range(n_iter):
        B = int(rng.integers(1, n_req + 1))
        sel = rng.permutation(n_req)[:B]
        ids, pos, rows = last_tok[sel], ctx[sel], tables[sel]
        # eager step (the request's K/V for this position is written; the replays below rewrite the same bits)
        logits_e, tok_e, _ = eng.step([1] * B, [int(p) for p in pos], ids, rows, list(range(B)))
        ref = bits(logits_e)
        tok_ref = tok_e.cpu().numpy().copy()
        small = graphs.bucket_for(B)
        for Bk in {small, buckets[-1]} | ({buckets[buckets.index(small) + 1]} if small != buckets[-1] else set()):
            logits_g, tok_g = graphs.step(ids, pos, rows, bucket=Bk)
            got = bits(logits_g)
            assert np.array_equal(got, ref), (it, B, Bk)
            assert np.array_equal(tok_g.cpu().numpy(), tok_ref), (it, B, Bk)
            checked += 1
        last_tok[sel] = tok_ref
        ctx[sel] += 1
    eng.check()
    graphs.close()
    eng.close()
    return checked


def test_tiny_graph_buckets_bitwise(mods):
    bi, Engine, DecodeGraphs = mods
    checked = run_fuzz(bi, Engine, DecodeGraphs, TINY, n_req=40, lo=1, hi=300, n_iter=24,
                       ladder=(1, 2, 4, 8, 16, 24, 32, 48), seed=5)
    assert checked >= 24


def test_8b_layer_graph_buckets_bitwise(mods):
    bi, Engine, DecodeGraphs = mods
    checked = run_fuzz(bi, Engine, DecodeGraphs, LLAMA3_8B_1L, n_req=20, lo=128, hi=2048, n_iter=6,
                       ladder=(1, 4, 8, 16, 24), seed=6)
    assert checked >= 6


def test_graph_rejects_positions_beyond_capture(mods):
    bi, Engine, DecodeGraphs = mods
    eng = Engine(TINY, num_pages=16, max_pages=4, max_T=8, max_B=4, max_R=8)
    g = DecodeGraphs(eng, 40, ladder=(1, 2))
    with pytest.raises(ValueError):
        g.step([1], [40], np.zeros((1, 4), np.int32))
    with pytest.raises(ValueError):
        g.step([1, 2, 3], [0, 0, 0], np.zeros((3, 4), np.int32))
    g.close()
    eng.close()
