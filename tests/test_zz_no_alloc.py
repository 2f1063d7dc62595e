"""The allocation-free decode attention entry point, against the allocating one.

cc_op_attention_decode_noalloc serves callers that cannot call cudaMalloc (a runtime whose
memory pool already owns the device, a decode loop that must not take cudaMalloc's
possible device-wide synchronisation, a host not allowed to allocate): its split-KV scratch
is a fixed array inside the library. This file is collected last so that a run stopping at
its first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import cohere_compass_decoder_gb300._lib as L

from gpu_util import require_gpu, bf16_dev, f64, assert_close

pytestmark = pytest.mark.gpu


def _problem(seed, B, nq, nkv, max_pages, window):
    rng = np.random.default_rng(seed)
    ps = 16
    n_pages = B * max_pages + 3
    n_keys = rng.integers(1, max_pages * ps + 1, size=B).astype(np.int32)
    table = rng.permutation(n_pages)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    return dict(
        q=bf16_dev(rng.standard_normal((B, nq * 128))),
        k=bf16_dev(rng.standard_normal((n_pages, nkv, ps, 128))),
        v=bf16_dev(rng.standard_normal((n_pages, nkv, ps, 128))),
        n_pages=n_pages, table=torch.from_numpy(table).cuda(), max_pages=max_pages,
        n_keys=torch.from_numpy(n_keys).cuda(), B=B, nq=nq, nkv=nkv, ps=ps, window=window)


def _run(fn, p, **extra):
    out = torch.full((p["B"], p["nq"] * 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    fn(p["q"], p["k"], p["v"], p["n_pages"], p["table"], p["max_pages"], p["n_keys"], p["B"],
       p["nq"], p["nkv"], p["ps"], p["window"], out, p["nq"] * 128, **extra)
    return out


def test_noalloc_decode_matches_allocating_entry_point():
    require_gpu()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # two calls in a row on different problems: the shared scratch keeps the first call's
    # contents, which must not leak into the second result
    for seed, (B, nq, nkv, max_pages, window) in ((1, (6, 16, 4, 33, 0)),
                                                  (2, (11, 8, 2, 20, 100))):
        p = _problem(seed, B, nq, nkv, max_pages, window)
        want = _run(L.cc_op_attention_decode, p)
        torch.cuda.synchronize()
        L.cc_op_sync()
        got = _run(L.cc_op_attention_decode_noalloc, p, err_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(f64(got), f64(want), 2e-2, 2e-3, "no-alloc decode attention")


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
