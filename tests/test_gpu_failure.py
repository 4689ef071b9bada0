"""Failure detection on the device, without a fault: a bounded wait that never
completes gives up after about a second, ORs the timeout bit into the
caller's error word and returns, rc_sync reports RC_ERR_TIMEOUT (and clears
the word), and the context keeps running kernels afterwards."""
from __future__ import annotations

import time

import pytest
import torch

import radixattention_prefix_shared_tree_gb300 as ra

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_the_context_stays_usable(cuda):
    err = torch.zeros(1, dtype=torch.int32, device=cuda)
    t0 = time.perf_counter()
    assert ra.rc_probe_wait_timeout(err) == ra.RC_OK
    assert ra.rc_sync(err) == ra.RC_ERR_TIMEOUT
    waited = time.perf_counter() - t0
    assert 0.2 < waited < 30.0          # the wait's limit is about one second
    assert ra.rc_sync(err) == ra.RC_OK  # the word was cleared

    # the same stream and context still run kernels: a scatter into a pool
    g = torch.Generator().manual_seed(5)
    n_slots, hkv, d, n = 64, 8, 128, 16
    k_pool = torch.zeros(n_slots, hkv, d, dtype=torch.bfloat16, device=cuda)
    v_pool = torch.zeros_like(k_pool)
    desc = ra.make_pool_desc(k_pool, v_pool, err)
    slots = torch.randperm(n_slots, generator=g)[:n].to(torch.int32).to(cuda)
    k = torch.randn(n, hkv, d, generator=g).to(torch.bfloat16).to(cuda)
    v = torch.randn(n, hkv, d, generator=g).to(torch.bfloat16).to(cuda)
    ra.kv_store(desc, slots, k, v)
    assert ra.rc_sync(err) == ra.RC_OK
    s = slots.long()
    assert torch.equal(k_pool[s], k) and torch.equal(v_pool[s], v)

