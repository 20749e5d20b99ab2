"""Forward-step tests through bi_forward_step:

* tiny single layer + LM head: oracle parity of every prompt position, and
  bitwise invariance over all 1500 splits of 8 requests into batches of 1, 2,
  4 and 8 (random in-batch order), prefill logits and decode logits;
* chunked prefill: any chunking of a prompt gives the same bits;
* the 8B-shaped layer: every request's layer output and logits bit-identical
  to its bs=1 run over random batch compositions of every size 1..64, oracle
  parity on a sample, and the batch-variant mode showing differences;
* a mixed continuous-batching fuzz (chunked prefill co-scheduled with
  decodes, arrival order, preemption, evict/readmit) on the 8B-shaped layer.
"""
import numpy as np
import pytest
import torch

import oracle
from invariant_fixed_order_gb300 import synth
from invariant_fixed_order_gb300.config import LLAMA3_8B_1L, TINY
from tests.helpers import assert_logits_close, f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from invariant_fixed_order_gb300 import bi, sched
    from invariant_fixed_order_gb300.engine import Engine
    return bi, sched, Engine


# ---------------------------------------------------------------------------
# tiny model
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def tiny(mods):
    bi, sched, Engine = mods
    eng = Engine(TINY, num_pages=1024, max_pages=24, max_T=8 * 260, max_B=8, max_R=8 * 260, keep_logical=True)
    lens = synth.uniform_ints(8, 1, 256, 42 + 0)
    prompts = [synth.token_ids(int(n), TINY.V, 500 + i) for i, n in enumerate(lens)]
    yield eng, prompts
    eng.close()


def run_block(sched, runner, prompts, rids, n_decode, rng=None, mode=None):
    """Prefill the block's prompts in one ragged step (all-position logits), then
    n_decode co-batched greedy decode steps.  Returns {rid: [positions, V]}."""
    reqs = [sched.Request(rid, prompts[rid]) for rid in rids]
    order = list(range(len(reqs))) if rng is None else list(rng.permutation(len(reqs)))
    out = {r.rid: [] for r in reqs}
    items = [sched.StepItem(reqs[i], len(reqs[i].prompt), "all") for i in order]
    logits, tokens, sl = runner.step(items, mode=mode)
    for it, s in zip(items, sl):
        out[it.req.rid].append(logits[s])
        it.req.generated.append(int(tokens[s][-1].item()))
    for _ in range(n_decode):
        order = list(range(len(reqs))) if rng is None else list(rng.permutation(len(reqs)))
        items = [sched.StepItem(reqs[i], 1, "last") for i in order]
        logits, tokens, sl = runner.step(items, mode=mode)
        for it, s in zip(items, sl):
            out[it.req.rid].append(logits[s])
            it.req.generated.append(int(tokens[s][0].item()))
    for r in reqs:
        runner.evict(r)
    return {rid: torch.cat(v) for rid, v in out.items()}


def test_tiny_oracle_parity(mods, tiny):
    bi, sched, _ = mods
    eng, prompts = tiny
    runner = sched.Runner(eng)
    dims = oracle.Dims(TINY.d, TINY.H, TINY.Hkv, TINY.Dh, TINY.F, TINY.eps, TINY.rope_theta)
    w = {k: f32(v) for k, v in eng.logical[0].items()}
    head = {k: f32(v) for k, v in eng.head.items()}
    got = run_block(sched, runner, prompts, list(range(8)), 0)
    eng.check()
    empty = [np.zeros((1, TINY.Hkv, TINY.Dh), np.float32)]
    for rid, p in enumerate(prompts):
        x = oracle.embed(head["embed"], p)
        x_out, _, _, _ = oracle.layer_forward(dims, w, [len(p)], [0], empty, empty, x)
        ref, ref_tok = oracle.lm_head(dims, head["gamma_final"], head["w_lm"], x_out, np.arange(len(p)))
        assert_logits_close(got[rid].cpu().numpy(), ref)


def test_tiny_all_partitions_bitwise(mods, tiny):
    """Every split of the 8 requests into batches of sizes 1/2/4/8, random order inside each batch."""
    bi, sched, _ = mods
    eng, prompts = tiny
    runner = sched.Runner(eng)
    n_decode = 2
    solo = {rid: run_block(sched, runner, prompts, [rid], n_decode)[rid] for rid in range(8)}
    rng = np.random.default_rng(1000)
    parts = list(sched.set_partitions_with_sizes(list(range(8)), {1, 2, 4, 8}))
    assert len(parts) == 1500
    ref = torch.cat([solo[r] for r in range(8)])
    n_checked = 0
    for part in parts:
        got = {}
        for block in part:
            got.update(run_block(sched, runner, prompts, block, n_decode, rng=rng))
        cat = torch.cat([got[r] for r in range(8)])
        if not sched.bitwise_equal(cat, ref):
            bad = [r for r in range(8) if not sched.bitwise_equal(got[r], solo[r])]
            pytest.fail(f"partition {part}: requests {bad} differ from their solo run: "
                        f"{[sched.diff_report(got[r], solo[r]) for r in bad]}")
        n_checked += 1
    eng.check()
    assert n_checked == 1500


def test_tiny_prefill_chunking_bitwise(mods, tiny):
    bi, sched, _ = mods
    eng, prompts = tiny
    runner = sched.Runner(eng)
    rid = int(np.argmax([len(p) for p in prompts]))
    p = prompts[rid]
    whole = run_block(sched, runner, prompts, [rid], 3)[rid]
    rng = np.random.default_rng(7)
    for trial in range(5):
        cuts = sorted(set(int(c) for c in rng.integers(1, len(p), size=trial + 1)))
        chunks = np.diff([0] + cuts + [len(p)]).tolist()
        req = sched.Request(rid, p)
        rows = []
        for n in chunks:
            logits, tokens, sl = runner.step([sched.StepItem(req, n, "all")])
            rows.append(logits[sl[0]])
        req.generated.append(int(tokens[sl[0]][-1].item()))
        for _ in range(3):
            logits, tokens, sl = runner.step([sched.StepItem(req, 1, "last")])
            rows.append(logits[sl[0]])
            req.generated.append(int(tokens[sl[0]][0].item()))
        runner.evict(req)
        assert sched.bitwise_equal(torch.cat(rows), whole), chunks


def test_tiny_greedy_tokens_follow_total_order(mods, tiny):
    """Greedy tokens of a forward step equal the total-order argmax of its
    logits, including exact ties (all LM-head rows equal: token 0) and NaN
    logits (two NaN rows: the lower index)."""
    bi, sched, _ = mods
    eng, prompts = tiny
    runner = sched.Runner(eng)
    w_lm = eng.head["w_lm"]
    saved = w_lm.clone()
    try:
        def run(rids):
            reqs = [sched.Request(rid, prompts[rid]) for rid in rids]
            items = [sched.StepItem(r, len(r.prompt), "all") for r in reqs]
            logits, tokens, _ = runner.step(items)
            out = (logits.clone(), tokens.clone())
            for r in reqs:
                runner.evict(r)
            return out
        logits, tokens = run([0, 3, 5])
        assert np.array_equal(tokens.cpu().numpy(), oracle.argmax_rows(logits.cpu().numpy()))
        w_lm.copy_(saved[7].expand_as(w_lm))
        logits, tokens = run([1, 2])
        assert bool((logits == logits[:, :1]).all())
        assert int(tokens.abs().sum()) == 0
        nan_row = saved[7].clone()
        nan_row[3] = float("nan")
        w_lm[700] = nan_row
        w_lm[1500] = nan_row
        logits, tokens = run([4])
        assert bool(torch.isnan(logits[:, 700]).all()) and bool(torch.isnan(logits[:, 1500]).all())
        assert bool((tokens == 700).all())
    finally:
        w_lm.copy_(saved)
        torch.cuda.synchronize()


def test_tiny_bad_token_reports_status(mods, tiny):
    """A token id outside the vocabulary is reported through the device status
    word (the embedding gather reads it as a zero row) and does not disturb
    the other requests of the step."""
    bi, sched, _ = mods
    eng, prompts = tiny
    good = [int(t) for t in prompts[2][:5]]
    table = np.zeros((2, eng.max_pages), np.int32)
    table[0, 0], table[1, 0] = eng.pool.alloc(1)[0], eng.pool.alloc(1)[0]
    try:
        ref, _, _ = eng.step([5], [0], good, table[:1], [4])
        ref = ref.clone()
        eng.check()
        logits, _, _ = eng.step([5, 3], [0, 0], good + [7, TINY.V + 3, 9], table, [4, 7])
        torch.cuda.synchronize()
        with pytest.raises(bi.BIError):
            eng.check()
        bi.reset_status(eng.status)
        assert torch.equal(logits[0], ref[0])
    finally:
        eng.pool.free([int(table[0, 0]), int(table[1, 0])])


def test_tiny_fused_final_norm_checks_replayed_logit_rows(mods, tiny):
    """With at most 8 logit rows that are the step's first tokens, the final RMSNorm runs inside the LM head on
    the residual stream's first R rows.  Device metadata (what a replay of such a captured step reads) must keep
    those rows: kept, the step gives the host-metadata step's bits; changed, the step reports
    BI_DEV_BAD_LOGIT_ROWS through the status word rather than answer silently for other rows."""
    bi, sched, _ = mods
    eng, prompts = tiny
    B = 3
    ids = [int(prompts[i][0]) for i in range(B)]
    table = np.zeros((B, eng.max_pages), np.int32)
    pages = [int(eng.pool.alloc(1)[0]) for _ in range(B)]
    table[:, 0] = pages
    try:
        ref, _, _ = eng.step([1] * B, [0] * B, ids, table, list(range(B)))
        ref = ref.clone()
        eng.check()
        d_ids = torch.tensor(ids, dtype=torch.int32, device="cuda")
        d_table = torch.from_numpy(table).cuda()
        for rows, ok in ((list(range(B)), True), ([2, 1, 0], False)):
            meta = torch.tensor(list(range(B)) + [0] * B + list(range(B)) + rows, dtype=torch.int32, device="cuda")
            logits = torch.empty(B, TINY.V, dtype=torch.float32, device="cuda")
            tokens = torch.empty(B, dtype=torch.int32, device="cuda")
            eng.model.forward_step([1] * B, [0] * B, d_ids, d_table, eng.k, eng.v, list(range(B)), eng.ws,
                                   eng.status, logits_out=logits, tokens_out=tokens, meta=meta)
            torch.cuda.synchronize()
            if ok:
                eng.check()
                assert torch.equal(logits.view(torch.int32), ref.view(torch.int32))
            else:
                with pytest.raises(bi.BIError) as e:
                    eng.check()
                assert "0x204" in str(e.value)
                bi.reset_status(eng.status)
    finally:
        eng.pool.free(pages)


# ---------------------------------------------------------------------------
# 8B-shaped single layer (decode steps over random compositions)
# ---------------------------------------------------------------------------

class DecodeLayerCase:
    """B requests with synthetic KV history (N(0,1)), contexts U[128, 8192]."""

    def __init__(self, Engine, n_req=64, seed=43):
        cfg = LLAMA3_8B_1L
        self.cfg = cfg
        self.ctx = synth.uniform_ints(n_req, 128, 8192, seed)
        self.ids = synth.token_ids(n_req, cfg.V, seed + 1)
        self.max_pages = 8192 // 16 + 1
        pages = int(sum((int(s) + 15) // 16 for s in self.ctx))
        self.eng = Engine(cfg, num_pages=pages + 64, max_pages=self.max_pages, max_T=n_req, max_B=n_req,
                          max_R=n_req, keep_logical=True)
        self.table = np.zeros((n_req, self.max_pages), np.int32)
        self.hist = []
        for i, s in enumerate(self.ctx):
            pg = self.eng.pool.alloc((int(s) + 15) // 16)
            self.table[i, :len(pg)] = pg
            k, v = synth.kv_history(int(s) - 1, cfg.Hkv, cfg.Dh, 7919 * seed + i, device="cuda")
            pos = np.arange(int(s) - 1)
            pt = torch.from_numpy(self.table[i, pos // 16].astype(np.int64)).cuda()
            sl = torch.from_numpy((pos % 16).astype(np.int64)).cuda()
            self.eng.k[0][pt, :, sl, :] = k
            self.eng.v[0][pt, :, sl, :] = v
            self.hist.append((k, v))
        self.d_table = torch.from_numpy(self.table).cuda()
        self.d_ids = torch.from_numpy(self.ids).cuda()

    def step(self, rows, mode):
        rows = list(rows)
        idx = torch.tensor(rows, device="cuda")
        logits, tokens, hidden = self.eng.step([1] * len(rows), [int(self.ctx[r]) - 1 for r in rows],
                                               self.d_ids[idx].contiguous(), self.d_table[idx].contiguous(),
                                               list(range(len(rows))), mode=mode, want_hidden=True)
        self.last_tokens = tokens
        return logits, hidden


@pytest.fixture(scope="module")
def layer8b(mods):
    bi, sched, Engine = mods
    case = DecodeLayerCase(Engine)
    yield case
    case.eng.close()


def test_8b_layer_compositions_bitwise(mods, layer8b):
    """Every batch size 1..64, 200 random compositions each: each request's layer
    output and logits are bit-identical to its bs=1 run."""
    bi, sched, _ = mods
    case = layer8b
    n = len(case.ctx)
    solo_l, solo_h, solo_t = [], [], []
    for r in range(n):
        l, h = case.step([r], bi.INVARIANT)
        solo_l.append(l[0].clone())
        solo_h.append(h[0].clone())
        solo_t.append(case.last_tokens[0].clone())
    solo_l = torch.stack(solo_l)
    solo_h = torch.stack(solo_h)
    solo_t = torch.stack(solo_t)
    # the greedy tokens (taken inside the LM head's epilogue) are the argmax of the logits
    assert np.array_equal(solo_t.cpu().numpy(), oracle.argmax_rows(solo_l.cpu().numpy()))
    rng = np.random.default_rng(1001)
    bad = 0
    for b in range(1, n + 1):
        for _ in range(200):
            rows = rng.choice(n, size=b, replace=False)
            l, h = case.step(rows, bi.INVARIANT)
            r = torch.from_numpy(rows).cuda()
            if not (sched.bitwise_equal(l, solo_l[r]) and sched.bitwise_equal(h, solo_h[r])
                    and torch.equal(case.last_tokens[:b], solo_t[r])):
                bad += 1
    case.eng.check()
    assert bad == 0, f"{bad} compositions differ from bs=1"


def test_8b_layer_oracle_parity(mods, layer8b):
    bi, sched, _ = mods
    case = layer8b
    cfg = case.cfg
    dims = oracle.Dims(cfg.d, cfg.H, cfg.Hkv, cfg.Dh, cfg.F, cfg.eps, cfg.rope_theta)
    w = {k: f32(v) for k, v in case.eng.logical[0].items()}
    gamma_final, w_lm = f32(case.eng.head["gamma_final"]), f32(case.eng.head["w_lm"])
    E = case.eng.head["embed"]
    rows = [int(np.argmin(case.ctx)), int(np.argmax(case.ctx)), 3, 17]
    # the full 64-request step, as the bench runs it; sampled rows checked one by one
    logits_all, hidden_all = case.step(range(len(case.ctx)), bi.INVARIANT)
    logits, hidden = logits_all[rows], hidden_all[rows]
    for j, r in enumerate(rows):
        k, v = case.hist[r]
        x = f32(E[int(case.ids[r])])[None]
        x_out, attn, _, _ = oracle.layer_forward(dims, w, [1], [int(case.ctx[r]) - 1], [f32(k)], [f32(v)], x)
        ref_logits, ref_tok = oracle.lm_head(dims, gamma_final, w_lm, x_out, [0])
        assert_logits_close(logits[j:j + 1].cpu().numpy(), ref_logits)
        # the layer output (bf16 residual stream) within a few bf16 ulps
        got_h = f32(hidden[j])
        assert np.max(np.abs(got_h - x_out[0])) <= 4 * 2.0 ** -8 * (np.max(np.abs(x_out[0])) + 1)


def test_8b_prefill_chunk_with_decodes_oracle_parity(mods, layer8b):
    """A 300-token prompt prefilled in the same step as four decode requests of the 8B-shaped layer (T = 304:
    256-wide GEMM tiles, RoPE over many positions in the QKV epilogue, tcgen05 prefill attention over two
    chunks): the logits of every prompt position and of the decode rows, and the layer output of every token,
    against the oracle."""
    bi, sched, _ = mods
    case = layer8b
    cfg = case.cfg
    dims = oracle.Dims(cfg.d, cfg.H, cfg.Hkv, cfg.Dh, cfg.F, cfg.eps, cfg.rope_theta)
    w = {k: f32(v) for k, v in case.eng.logical[0].items()}
    gamma_final, w_lm = f32(case.eng.head["gamma_final"]), f32(case.eng.head["w_lm"])
    E = case.eng.head["embed"]
    n = 300
    T = n + 4
    prompt = synth.token_ids(n, cfg.V, 777)
    pages = case.eng.pool.alloc((n + 15) // 16)
    ws_small = case.eng.ws
    case.eng.ws = torch.empty(case.eng.model.workspace_size(T, 5, T, case.eng.max_seq), dtype=torch.uint8,
                              device="cuda")
    try:
        prow = np.zeros(case.max_pages, np.int32)
        prow[:len(pages)] = pages
        dec = [3, int(np.argmin(case.ctx)), 17, int(np.argmax(case.ctx))]
        # decode, decode, the prompt, decode, decode
        q_len = [1, 1, n, 1, 1]
        pos0 = [int(case.ctx[dec[0]]) - 1, int(case.ctx[dec[1]]) - 1, 0, int(case.ctx[dec[2]]) - 1,
                int(case.ctx[dec[3]]) - 1]
        ids = np.concatenate([case.ids[dec[:2]], prompt, case.ids[dec[2:]]]).astype(np.int32)
        table = np.stack([case.table[dec[0]], case.table[dec[1]], prow, case.table[dec[2]], case.table[dec[3]]])
        logits, _, hidden = case.eng.step(q_len, pos0, ids, table, list(range(T)), want_hidden=True)
        case.eng.check()
        logits, hidden = logits.cpu().numpy(), f32(hidden)
        # the prompt: every position
        x = f32(E[torch.from_numpy(prompt.astype(np.int64)).cuda()])
        empty = [np.zeros((1, cfg.Hkv, cfg.Dh), np.float32)]
        x_out, _, _, _ = oracle.layer_forward(dims, w, [n], [0], empty, empty, x)
        ref_logits, _ = oracle.lm_head(dims, gamma_final, w_lm, x_out, np.arange(n))
        got = logits[2:2 + n]
        assert_logits_close(got, ref_logits)
        row_err = np.max(np.abs(got - ref_logits), axis=1)
        assert np.all(row_err <= 2e-2 * np.max(np.abs(ref_logits), axis=1))
        assert np.max(np.abs(hidden[2:2 + n] - x_out)) <= 4 * 2.0 ** -8 * (np.max(np.abs(x_out)) + 1)
        # the decode rows
        for j, (r, t) in enumerate(zip(dec, (0, 1, n + 2, n + 3))):
            k, v = case.hist[r]
            xd = f32(E[int(case.ids[r])])[None]
            xd_out, _, _, _ = oracle.layer_forward(dims, w, [1], [int(case.ctx[r]) - 1], [f32(k)], [f32(v)], xd)
            ref_d, _ = oracle.lm_head(dims, gamma_final, w_lm, xd_out, [0])
            assert_logits_close(logits[t:t + 1], ref_d)
            assert np.max(np.abs(hidden[t] - xd_out[0])) <= 4 * 2.0 ** -8 * (np.max(np.abs(xd_out[0])) + 1)
    finally:
        case.eng.ws = ws_small
        case.eng.pool.free(pages)


def test_8b_layer_variant_mode_negative_control(mods, layer8b):
    """Variant mode must show bit differences against bs=1 somewhere (the
    harness has teeth), stay within the parity tolerance, and repeat itself on
    an identical batch (determinism at fixed batch)."""
    bi, sched, _ = mods
    case = layer8b
    n = len(case.ctx)
    solo = torch.stack([case.step([r], bi.VARIANT)[0][0].clone() for r in range(n)])
    rng = np.random.default_rng(1002)
    diffs = checked = 0
    for b in (2, 4, 8, 16, 32, 64):
        for _ in range(4):
            rows = rng.choice(n, size=b, replace=False)
            l, _ = case.step(rows, bi.VARIANT)
            ref = solo[torch.from_numpy(rows).cuda()]
            for j in range(b):
                checked += 1
                if not sched.bitwise_equal(l[j], ref[j]):
                    diffs += 1
            err = (l - ref).abs().max().item()
            assert err <= 2e-2 * ref.abs().max().item()
    again, _ = case.step(rows, bi.VARIANT)
    assert sched.bitwise_equal(again, l)
    assert diffs > 0, f"batch-variant mode never differed in {checked} rows: the harness would have no teeth"


# ---------------------------------------------------------------------------
# mixed continuous batching on the 8B-shaped layer
# ---------------------------------------------------------------------------

def test_8b_continuous_batching_fuzz(mods):
    """Chunked prefill (256-2048) co-scheduled with decode requests (contexts
    up to 32768), random arrival order, preemption and evict/readmit: every
    produced logits row equals the solo run bit for bit."""
    bi, sched, Engine = mods
    cfg = LLAMA3_8B_1L
    rng = np.random.default_rng(1003)
    long_lens = rng.integers(512, 32768, 3)  # decode contexts up to 32768 positions
    long_lens[0] = 32760
    short_lens = rng.integers(256, 2048, 3)
    lens = [int(x) for x in np.concatenate([long_lens, short_lens])]
    prompts = [synth.token_ids(n, cfg.V, 900 + i) for i, n in enumerate(lens)]
    n_decode = 4
    max_pages = (max(lens) + n_decode + 15) // 16 + 1
    eng = Engine(cfg, num_pages=sum(lens) // 16 + 64 * len(lens), max_pages=max_pages,
                 max_T=max(max(lens), 4096) + 64, max_B=16, max_R=16)
    runner = sched.Runner(eng)
    solo = {}
    teacher = {}
    for rid, p in enumerate(prompts):
        req = sched.Request(rid, p)
        # solo: the whole prompt in one prefill, then greedy decode, alone
        out = {}
        logits, tokens, sl = runner.step([sched.StepItem(req, len(p), "last")])
        out[len(p) - 1] = logits[sl[0]][0].clone()
        for _ in range(n_decode):
            req.generated.append(int(tokens[sl[0]][-1].item()))
            if len(req.generated) > n_decode - 1:
                break
            logits, tokens, sl = runner.step([sched.StepItem(req, 1, "last")])
            out[req.n_cached - 1] = logits[sl[0]][0].clone()
        teacher[rid] = list(req.generated)
        solo[rid] = out
        runner.evict(req)
    eng.check()
    fz = sched.FuzzConfig(token_budget=4096, chunk_min=256, chunk_max=2048, p_evict=0.15, readmit_delay=(1, 3),
                          arrival_span=4)
    for trial in range(6):
        reqs = [sched.Request(rid, p) for rid, p in enumerate(prompts)]
        got = sched.fuzz_continuous(runner, reqs, n_decode, np.random.default_rng(2000 + trial), fz,
                                    teacher=teacher, all_prompt_logits=False)
        eng.check()
        for rid in range(len(prompts)):
            for pos, row in solo[rid].items():
                assert pos in got[rid], (trial, rid, pos, sorted(got[rid]))
                assert sched.bitwise_equal(got[rid][pos], row), (trial, rid, pos,
                                                                  sched.diff_report(got[rid][pos], row))
    eng.close()
