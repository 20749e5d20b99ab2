"""System tests on multi-layer 8B-shaped models (random weights):

* unique completions: every prompt decoded greedily under several randomised
  continuous-batching schedules (random arrival, batch composition, chunked
  prefill, evict/readmit) gives exactly one completion, equal to its solo run
  (and the 95% rule-of-three bound on the divergence rate is reported);
* decode-verify-rollback: the batch-variant fast path verified by invariant
  replay commits exactly the pure invariant greedy tokens, including when the
  fast path is forced to emit wrong candidates.

Sizes are reduced from the full configurations so the suite stays within
minutes; BI_SYSTEM_SCALE=full runs the full ones (32 layers, 64 prompts of
128-4096 tokens, 256 generated tokens, 50 schedules)."""
import os
import time

import numpy as np
import pytest
import torch

from invariant_fixed_order_gb300 import results, synth
from invariant_fixed_order_gb300.config import LLAMA3_8B

pytestmark = pytest.mark.gpu

FULL = os.environ.get("BI_SYSTEM_SCALE") == "full"


@pytest.fixture(scope="module")
def mods():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from invariant_fixed_order_gb300 import bi, dvr, sched
    from invariant_fixed_order_gb300.engine import Engine
    return bi, sched, dvr, Engine


def greedy_solo(sched, runner, prompt, rid, n_new, mode):
    req = sched.Request(rid, prompt)
    logits, tokens, sl = runner.step([sched.StepItem(req, len(prompt), "last")], mode=mode)
    req.generated.append(int(tokens[sl[0]][-1].item()))
    while len(req.generated) < n_new:
        logits, tokens, sl = runner.step([sched.StepItem(req, 1, "last")], mode=mode)
        req.generated.append(int(tokens[sl[0]][0].item()))
    runner.evict(req)
    return list(req.generated)


def greedy_batched(sched, runner, prompts, n_new, mode):
    """Greedy decoding of all prompts together (prompts prefilled one by one)."""
    reqs = [sched.Request(rid, p) for rid, p in enumerate(prompts)]
    for r in reqs:
        logits, tokens, sl = runner.step([sched.StepItem(r, len(r.prompt), "last")], mode=mode)
        r.generated.append(int(tokens[sl[0]][-1].item()))
    while len(reqs[0].generated) < n_new:
        logits, tokens, sl = runner.step([sched.StepItem(r, 1, "last") for r in reqs], mode=mode)
        tok = tokens.tolist()
        for r, s_ in zip(reqs, sl):
            r.generated.append(tok[s_.start])
    out = {r.rid: list(r.generated) for r in reqs}
    for r in reqs:
        runner.evict(r)
    return out


def test_unique_completions_under_random_schedules(mods):
    bi, sched, dvr, Engine = mods
    n_layers, n_prompts, lo, hi, n_new, n_sched = (32, 64, 128, 4096, 256, 50) if FULL else (16, 24, 128, 1024, 40, 6)
    cfg = LLAMA3_8B.with_layers(n_layers)
    lens = [int(x) for x in synth.uniform_ints(n_prompts, lo, hi, 42 + 4)]
    prompts = [synth.token_ids(n, cfg.V, 4000 + i) for i, n in enumerate(lens)]
    max_pages = (hi + n_new + 15) // 16 + 1
    eng = Engine(cfg, num_pages=sum((n + n_new + 15) // 16 + 1 for n in lens) + 256, max_pages=max_pages,
                 max_T=max(4096, hi) + n_prompts, max_B=n_prompts, max_R=n_prompts)
    runner = sched.Runner(eng)
    solo = {rid: greedy_solo(sched, runner, p, rid, n_new, bi.INVARIANT) for rid, p in enumerate(prompts)}
    completions = {rid: {tuple(solo[rid])} for rid in solo}
    # an eviction frees the request's pages; its readmission recomputes up to 4k positions through every
    # layer by chunked prefill (at full size ~80 evictions per schedule)
    fz = sched.FuzzConfig(token_budget=4096, chunk_min=256, chunk_max=2048, p_evict=0.005 if FULL else 0.05,
                          readmit_delay=(1, 3), arrival_span=6)
    counts = {}
    t_start = time.perf_counter()
    print(f"unique completions: {n_layers} layers, {n_prompts} prompts, {n_new} tokens, {n_sched} schedules",
          flush=True)
    for k in range(n_sched):
        reqs = [sched.Request(rid, p) for rid, p in enumerate(prompts)]
        sched.fuzz_continuous(runner, reqs, n_new, np.random.default_rng(1000 + k), fz, all_prompt_logits=False,
                              stats=counts)
        eng.check()
        for r in reqs:
            completions[r.rid].add(tuple(r.generated[:n_new]))
        print(f"  schedule {k}: max completions per prompt so far {max(len(c) for c in completions.values())}",
              flush=True)
    unique = {rid: len(c) for rid, c in completions.items()}
    bound = sched.rule_of_three(n_prompts * n_sched)
    print(f"unique completions per prompt: max {max(unique.values())}; rule-of-three bound {bound:.4f}; "
          f"{counts}")
    results.record("unique_completions" + ("_full" if FULL else ""), {
        "mode": "invariant", "layers": n_layers, "prompts": n_prompts, "prompt_len": [lo, hi], "new_tokens": n_new,
        "schedules": n_sched, "seeds": {"prompt_lengths": 42 + 4, "prompt_tokens": "4000 + i", "weights": 1234,
                                        "schedules": "1000 + k"},
        "fuzz": {"token_budget": fz.token_budget, "chunk": [fz.chunk_min, fz.chunk_max], "p_evict": fz.p_evict,
                 "readmit_delay": list(fz.readmit_delay), "arrival_span": fz.arrival_span},
        "counts": counts, "max_completions_per_prompt": max(unique.values()),
        "prompts_with_one_completion": sum(1 for u in unique.values() if u == 1),
        "divergent_trials": sum(u - 1 for u in unique.values()), "trials": n_prompts * n_sched,
        "rule_of_three_bound": bound, "seconds": round(time.perf_counter() - t_start, 1)})
    assert all(u == 1 for u in unique.values()), unique
    eng.close()


def test_decode_throughput_invariant_vs_variant(mods):
    """Greedy decode throughput of the multi-layer model at batch 64 (and 1),
    invariant vs batch-variant mode (reported; variant is the faster one)."""
    bi, sched, dvr, Engine = mods
    n_layers, n_prompts, n_steps = (32, 64, 64) if FULL else (8, 64, 16)
    cfg = LLAMA3_8B.with_layers(n_layers)
    lens = [int(x) for x in synth.uniform_ints(n_prompts, 128, 4096, 42 + 6)]
    max_pages = (4096 + n_steps + 15) // 16 + 1
    eng = Engine(cfg, num_pages=sum((n + n_steps + 15) // 16 + 1 for n in lens) + 64, max_pages=max_pages,
                 max_T=max(lens) + 64, max_B=n_prompts, max_R=n_prompts)
    runner = sched.Runner(eng)
    out = {}
    for mode_name, mode in (("invariant", bi.INVARIANT), ("variant", bi.VARIANT)):
        for b in (1, n_prompts):
            reqs = [sched.Request(i, synth.token_ids(lens[i], cfg.V, 6000 + i)) for i in range(b)]
            for r in reqs:  # prompts prefilled one by one (not timed)
                logits, tokens, sl = runner.step([sched.StepItem(r, len(r.prompt), "last")], mode=mode)
                r.generated.append(int(tokens[sl[0]][-1].item()))
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(n_steps):
                items = [sched.StepItem(r, 1, "last") for r in reqs]
                logits, tokens, sl = runner.step(items, mode=mode)
                tok = tokens.tolist()
                for r, s_ in zip(reqs, sl):
                    r.generated.append(tok[s_.start])
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / n_steps
            out[f"{mode_name}_bs{b}"] = {"ms_per_step": round(ms, 3), "tok_s": round(b / (ms * 1e-3), 1)}
            for r in reqs:
                runner.evict(r)
    eng.check()
    print(f"decode throughput, {n_layers} layers (host scheduler in the loop):", out)
    assert out[f"variant_bs{n_prompts}"]["tok_s"] > 0 and out[f"invariant_bs{n_prompts}"]["tok_s"] > 0
    eng.close()


def test_decode_verify_rollback_commits_the_invariant_greedy_tokens(mods):
    bi, sched, dvr, Engine = mods
    n_layers, n_prompts, n_new, window = (32, 64, 256, 64) if FULL else (8, 16, 96, 32)
    cfg = LLAMA3_8B.with_layers(n_layers)
    lens = [int(x) for x in synth.uniform_ints(n_prompts, 128, 1024, 42 + 5)]
    prompts = [synth.token_ids(n, cfg.V, 5000 + i) for i, n in enumerate(lens)]
    max_pages = (1024 + n_new + window + 15) // 16 + 1
    eng = Engine(cfg, num_pages=n_prompts * max_pages + 64, max_pages=max_pages,
                 max_T=max(8 * window, 8 * 1024) + 64, max_B=n_prompts, max_R=8 * window)
    runner = sched.Runner(eng)
    # pure invariant greedy decoding (batched: invariant mode gives every request its solo bits)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    truth = greedy_batched(sched, runner, prompts, n_new, bi.INVARIANT)
    torch.cuda.synchronize()
    t_invariant = time.perf_counter() - t0

    # plain run of the fast path
    reqs = [sched.Request(rid, p) for rid, p in enumerate(prompts)]
    st = dvr.dvr_generate(runner, reqs, n_new, window=window, verify_batch=8)
    eng.check()
    for r in reqs:
        assert r.generated == truth[r.rid], r.rid
        runner.evict(r)
    assert st.committed == n_prompts * n_new
    summary = st.as_dict(window=window)
    summary["invariant_greedy_tok_s"] = n_prompts * n_new / t_invariant
    summary["committed_vs_invariant"] = summary["committed_tok_s"] / summary["invariant_greedy_tok_s"]
    print(f"dvr ({n_layers} layers, {n_prompts} prompts, {n_new} tokens, window {window}):", summary, flush=True)
    results.record("dvr" + ("_full" if FULL else ""), {
        "layers": n_layers, "prompts": n_prompts, "prompt_len": [128, 1024], "new_tokens": n_new, "window": window,
        "verify_batch": 8, "fast_mode": "variant", "verifier": "invariant teacher-forced replay",
        "seeds": {"prompt_lengths": 42 + 5, "prompt_tokens": "5000 + i", "weights": 1234},
        "committed_equals_invariant_greedy": True, "stats": summary})

    # a fast path that emits wrong candidates at chosen positions: the verifier
    # must catch each one, roll back and still commit exactly the greedy tokens
    bad = {(rid, len(prompts[rid]) + 5 + 7 * rid) for rid in range(n_prompts)}
    reqs = [sched.Request(rid, p) for rid, p in enumerate(prompts)]
    st2 = dvr.dvr_generate(runner, reqs, n_new, window=window, verify_batch=8,
                           corrupt=lambda rid, pos: (rid, pos) in bad)
    eng.check()
    for r in reqs:
        assert r.generated == truth[r.rid], r.rid
        runner.evict(r)
    assert st2.mismatched_windows >= n_prompts
    assert st2.rollback_rate > 0
    eng.close()


def test_dvr_per_request_opt_in_and_tuning(mods):
    """"Per-Request Opt-In and Mixed Workloads": only requests marked deterministic are verified; they
    commit exactly the pure invariant greedy tokens while sharing fast-path batches with unverified
    requests, and the verifier's work covers only them.  Window and verify-batch sizes are swept
    ("The window size and verify batch size are tunable parameters")."""
    bi, sched, dvr, Engine = mods
    n_layers, n_prompts, n_new = (8, 16, 48)
    cfg = LLAMA3_8B.with_layers(n_layers)
    lens = [int(x) for x in synth.uniform_ints(n_prompts, 128, 768, 42 + 7)]
    prompts = [synth.token_ids(n, cfg.V, 6000 + i) for i, n in enumerate(lens)]
    max_pages = (768 + n_new + 64 + 15) // 16 + 1
    eng = Engine(cfg, num_pages=n_prompts * max_pages + 64, max_pages=max_pages,
                 max_T=16 * 768 + 64, max_B=n_prompts, max_R=16 * 64)
    runner = sched.Runner(eng)
    truth = greedy_batched(sched, runner, prompts, n_new, bi.INVARIANT)
    det = {rid for rid in range(n_prompts) if rid % 2 == 0}
    results = {}
    for window, vb in ((16, 4), (32, 8), (48, 16)):
        reqs = [sched.Request(rid, p, is_deterministic=rid in det) for rid, p in enumerate(prompts)]
        st = dvr.dvr_generate(runner, reqs, n_new, window=window, verify_batch=vb)
        eng.check()
        for r in reqs:
            assert len(r.generated) == n_new, r.rid
            if r.is_deterministic:
                assert r.generated == truth[r.rid], r.rid
            runner.evict(r)
        # every verified window belongs to a deterministic request
        assert st.verified == det, st.verified
        assert st.windows >= len(det) * (-(-(n_new - 1) // window))
        results[(window, vb)] = st.as_dict()
    print("dvr opt-in (8 layers, 16 prompts, half deterministic):", results, flush=True)
    eng.close()
