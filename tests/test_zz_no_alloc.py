"""The allocation-free decode attention entry point, against the allocating one and the oracle.

cc_op_attention_decode_noalloc serves callers that cannot call cudaMalloc (a runtime whose
memory pool already owns the device, a decode loop that must not take cudaMalloc's
possible device-wide synchronisation, a host not allowed to allocate): its split-KV scratch
is a fixed array inside the library, shared by every call and never cleared. Both entry
points run the same kernels on the same inputs, so their outputs must be bit-identical;
anything less would mean that the shared scratch leaked one call's partials into another.
This file is collected last so that a run stopping at its first failure has already run
every other test.
"""
import numpy as np
import pytest
import torch

import cohere_compass_decoder_gb300._lib as L
from oracle import decoder as O

from gpu_util import require_gpu, bf16_dev, f64, assert_close

pytestmark = pytest.mark.gpu

PS = 16


def _problem(seed, B, nq, nkv, max_pages, window, n_keys):
    rng = np.random.default_rng(seed)
    n_pages = B * max_pages + 3
    table = rng.permutation(n_pages)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    return dict(
        q=bf16_dev(rng.standard_normal((B, nq * 128))),
        k=bf16_dev(rng.standard_normal((n_pages, nkv, PS, 128))),
        v=bf16_dev(rng.standard_normal((n_pages, nkv, PS, 128))),
        n_pages=n_pages, table=torch.from_numpy(table).cuda(),
        max_pages=max_pages, n_keys_np=np.asarray(n_keys, np.int32),
        n_keys=torch.from_numpy(np.asarray(n_keys, np.int32)).cuda(), B=B, nq=nq, nkv=nkv,
        window=window)


def _run(fn, p, **extra):
    out = torch.full((p["B"], p["nq"] * 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    fn(p["q"], p["k"], p["v"], p["n_pages"], p["table"], p["max_pages"], p["n_keys"], p["B"],
       p["nq"], p["nkv"], PS, p["window"], out, p["nq"] * 128, **extra)
    return out


def _oracle(p, rows):
    """Decode attention of the sequences `rows` by the oracle: the query is the last of the
    sequence's n_keys tokens, keys gathered through the page table."""
    Q = f64(p["q"]).reshape(p["B"], p["nq"], 128)
    want = np.zeros((len(rows), p["nq"], 128))
    for r, b in enumerate(rows):
        n = int(p["n_keys_np"][b])
        idx = torch.arange(n, device="cuda")
        pages = p["table"][b][idx // PS].long()
        K = f64(p["k"][pages, :, idx % PS, :])      # [n, nkv, 128], gathered on the device
        V = f64(p["v"][pages, :, idx % PS, :])
        want[r] = O.decode_attention(Q[b], K, V, p["window"] if p["window"] > 0 else None,
                                     128 ** -0.5)
    return want


def _both(p, err):
    want = _run(L.cc_op_attention_decode, p)
    torch.cuda.synchronize()
    L.cc_op_sync()
    got = _run(L.cc_op_attention_decode_noalloc, p, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return got, want


def test_noalloc_decode_two_calls_many_splits_then_mostly_empty_splits():
    """Call 1 fills every split of a 300-page problem (5 splits of 64 pages); call 2 has the
    same scratch layout but few keys (or a short window), so most of its splits are empty and
    must mark themselves so instead of merging call 1's partials still in the scratch."""
    require_gpu()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B, nq, nkv, max_pages = 8, 16, 4, 300
    rng = np.random.default_rng(7)
    full = rng.integers(max_pages * PS - 120, max_pages * PS + 1, size=B)
    few = rng.integers(1, 200, size=B)
    few[0] = 1
    cases = ((11, 0, full), (12, 0, few), (13, 0, full), (14, 96, full))
    for seed, window, n_keys in cases:
        p = _problem(seed, B, nq, nkv, max_pages, window, n_keys)
        got, want = _both(p, err)
        assert torch.equal(got, want), f"no-alloc differs from the allocating call (seed {seed})"
        assert_close(f64(got).reshape(B, nq, 128), _oracle(p, range(B)), 2e-2, 2e-3,
                     f"no-alloc decode attention vs oracle (seed {seed})")


def test_noalloc_decode_at_the_benchmarked_shape():
    """64 sequences x 4097 keys (4096 cached + the new one), 16 / 4 heads, 257-page table:
    sliding (window 4096) and full, twice in a row each."""
    require_gpu()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B, nq, nkv, max_pages = 64, 16, 4, 257
    for seed, window in ((21, 4096), (22, 0), (23, 4096)):
        p = _problem(seed, B, nq, nkv, max_pages, window, np.full(B, 4097))
        got, want = _both(p, err)
        assert torch.equal(got, want), f"no-alloc differs from the allocating call (seed {seed})"
        rows = [0, 17, 40, 63]
        assert_close(f64(got).reshape(B, nq, 128)[rows], _oracle(p, rows), 2e-2, 2e-3,
                     f"no-alloc decode attention vs oracle (seed {seed})")


def test_noalloc_decode_rejects_problems_beyond_its_scratch():
    require_gpu()
    # 64 sequences x 16 heads x 300 splits x 130 floats > 4 Mi floats
    B, nq, nkv, max_pages = 64, 16, 4, 16 * 300
    q = torch.zeros(B, nq * 128, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(1, nkv, 16, 128, dtype=torch.bfloat16, device="cuda")
    table = torch.zeros(B, max_pages, dtype=torch.int32, device="cuda")
    nk = torch.ones(B, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(L.CCError) as e:
        L.cc_op_attention_decode_noalloc(q, kv, kv, 1, table, max_pages, nk, B, nq, nkv, 16, 0,
                                         out, nq * 128)
    assert e.value.status == L.CC_ERR_INVALID_ARG
