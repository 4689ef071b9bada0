"""Token-granular radix tree vs 16-token block cache on the same traces.

"RadixAttention, eviction and cache churn" (inference-notes note 49),
section 3, compares RadixAttention's token-granular matching with vLLM's
prefix caching over a hash chain of 16-token blocks: same sharing by
reference count, same least-recently-used eviction, different match
granularity.  This replays each workload's host side (admission in
scheduling order, eviction, insert after prefill, insert of prompt + outputs
at finish) through both caches of the library and reports, per cache, the
token hit rate (matched / prompt tokens), the request hit rate (matched > 0),
the tokens prefill must compute, evictions and the host time per request.

    python -m radixattention_prefix_shared_tree_gb300.compare [--json]
"""
from __future__ import annotations

import argparse
import json
import time

import numpy as np

from . import RC_LPM, BlockCache, RadixCache, rc_image_key
from . import workloads as wl


def _replay(name, make_cache, pool, trace, run):
    from synth.model import SynthModel
    cache = make_cache(pool)
    runner = wl.Runner(cache, SynthModel(trace.shape, trace.seed, trace.vocab, device="cpu"), engine=None,
                       policy=RC_LPM)
    served = []
    orig = runner.serve

    def serve(pending, max_batch=None):
        admitted, waiting = orig(pending, max_batch)
        served.extend(admitted)
        return admitted, waiting

    runner.serve = serve
    t0 = time.perf_counter()
    run(runner, trace)
    dt = time.perf_counter() - t0
    prompt = sum(r.prompt_len for r in served)
    matched = sum(r.matched for r in served)
    computed = sum(r.prompt_len - r.first for r in served)
    st = cache.stats()
    return {"requests": len(served), "prompt_tokens": prompt, "matched_tokens": matched,
            "token_hit_rate": matched / max(prompt, 1),
            "request_hit_rate": sum(1 for r in served if r.matched > 0) / max(len(served), 1),
            "prefill_tokens": computed, "evicted_tokens": st["evicted_tokens"],
            "host_us_per_request": 1e6 * dt / max(len(served), 1)}


def workloads():
    from synth import traces
    few = traces.few_shot()
    chat = traces.chat()
    agent = traces.agent_tree()
    mm = traces.multimodal()
    return [
        ("few-shot: 1792-token shared prefix, 256 questions U[32,64]", few, few.pool_slots or (1 << 21),
         lambda r, t: wl.run_few_shot(r, t)),
        ("chat: 256 sessions x 8 turns, pool 0.75 of the working set", chat, chat.pool_slots,
         lambda r, t: wl.run_chat(r, t)),
        ("agent tree: 2048 root, 4-way branching to depth 3, 256 per branch", agent, agent.pool_slots,
         lambda r, t: wl.run_agent(r, t)),
        ("multimodal: 50-token system, 24 images x 8 questions, 576 image keys each, rounds of 16", mm, mm.pool_slots,
         lambda r, t: wl.run_multimodal(r, t, rc_image_key, batch=16)),
    ]


def reuse_by_shared_length(block_tokens: int = 16, lengths=range(0, 65)) -> list:
    """Tokens a second prompt reuses when it shares its first L tokens with a
    cached one (the comparison of section 3), measured on both caches."""
    rng = np.random.default_rng(0)
    out = []
    for L in lengths:
        a = rng.integers(0, 1000, 96).astype(np.int32)
        b = np.concatenate([a[:L], [1000 + L], rng.integers(0, 1000, 8)]).astype(np.int32)
        row = {"shared": int(L)}
        for key, cache in (("radix", RadixCache(256)), (f"block{block_tokens}", BlockCache(256, block_tokens))):
            st, m, ms, node = cache.match(a, True)
            st, new = cache.alloc(len(a) - m)
            cache.insert(a, np.concatenate([ms, new]).astype(np.int32), False)
            row[key] = int(cache.match(b, False)[1])
        out.append(row)
    return out


def compare(block_tokens: int = 16) -> list:
    rows = []
    for name, trace, pool, run in workloads():
        rows.append({"workload": name,
                     "radix": _replay(name, RadixCache, pool, trace, run),
                     f"block{block_tokens}": _replay(name, lambda n: BlockCache(n, block_tokens), pool, trace,
                                                     run)})
    return rows


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--block-tokens", type=int, default=16)
    ap.add_argument("--json", action="store_true")
    a = ap.parse_args(argv)
    rows = compare(a.block_tokens)
    stair = reuse_by_shared_length(a.block_tokens)
    if a.json:
        print(json.dumps({"workloads": rows, "reuse_by_shared_length": stair}))
        return
    key = f"block{a.block_tokens}"
    print("reused tokens vs shared prefix length L (radix / block):",
          " ".join(f"{r['shared']}:{r['radix']}/{r[key]}" for r in stair if r["shared"] % 8 == 0 or
                   r["shared"] % 16 == 15))
    for r in rows:
        print(r["workload"])
        for k in ("radix", key):
            v = r[k]
            print(f"  {k:8s} token hit {v['token_hit_rate']:.4f}  request hit {v['request_hit_rate']:.3f}  "
                  f"prefill {v['prefill_tokens']:9d}  evicted {v['evicted_tokens']:8d}  "
                  f"host {v['host_us_per_request']:7.1f} us/request")


if __name__ == "__main__":
    main()
