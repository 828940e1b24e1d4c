"""GPU parity of the fused attention forward (hgemm_attention_*) with the oracle.

O = softmax(scale * Q K^T [causal]) V, head dimension 128, fp16 / bf16.
Bound: the kernel's scores and softmax are fp32 and its accumulation of P V
is fp32, but the probabilities are rounded to the input type before the
second product (as the pages' register hand-over of P does) and O is
rounded once.  With u the unit roundoff of the type (2^-8 for bf16's 8
significant bits, 2^-11 for fp16's 11) each of the two roundings moves O by at most u * sum_j p_j |v_j| / l
(the oracle's Den), so

    max |O - Oref| / Den <= 2u (+ ex2's 2^-22 and fp32 sums, far smaller),

and the test bound is 2.5u: 9.8e-3 for bf16, 1.2e-3 for fp16.  The scores
carry their own fp32 error: a sum of head_dim products is off by at most
g = head_dim * 2^-23 * sden (sden = max_j scale * sum |q||k| from the
oracle; 2^-23 allows truncating accumulation), which moves each p_j by a
factor within e^(+-g), so O by at most 2g * Den; the bound of a row is
2.5u + 2.5g.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tensor_core_dense_swizzled_gb300 import hgemm as H
from test_gpu_parity import dev  # noqa: F401 (fixture)

pytestmark = pytest.mark.gpu

D = 128
DT = {"bf16": H.HGEMM_BF16, "f16": H.HGEMM_F16}
TD = {"bf16": torch.bfloat16, "f16": torch.float16}
OC = {"bf16": oracle.BF16, "f16": oracle.F16}
TOL = {"bf16": 2.5 * 2.0 ** -8, "f16": 2.5 * 2.0 ** -11}


def bits(t):
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16).reshape(-1)


def draw(shape, seed, dt, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(TD[dt])


def run_attention(dev, q, k, v, bh, sq, skv, scale, causal, dt, runs=1):
    O = torch.full((bh * sq * D + 64,), 77.0, dtype=TD[dt], device=dev)
    plan = H.hgemm_attention_plan_create(bh, sq, skv, D, scale, causal, DT[dt])
    outs = []
    try:
        dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
        for _ in range(runs):
            H.hgemm_attention_run(plan, dq, dk, dv, O)
            st = H.hgemm_attention_check(plan)
            assert st == 0, f"{H.STATUS.get(st)} {H.hgemm_last_error_detail()}"
            outs.append(O.clone())
    finally:
        H.hgemm_attention_plan_destroy(plan)
    for o in outs[1:]:
        assert torch.equal(o, outs[0]), "repeated runs differ"
    assert torch.all(O[bh * sq * D:].cpu() == 77.0), "kernel wrote past the end of O"
    return O[: bh * sq * D].cpu()


def check(got, q, k, v, bh, sq, skv, scale, causal, dt, rows=None):
    Oref, Den, _, sden = oracle.attention(bits(q), bits(k), bits(v), OC[dt], bh, sq, skv, D, scale,
                                          causal, rows=rows)
    g = got.double().numpy().reshape(bh, sq, D)
    if rows is not None:
        g = g[rows[0], rows[1]]
    row_err = np.max(np.abs(g - Oref) / np.maximum(Den, 1e-300), axis=-1)
    row_tol = TOL[dt] + 2.5 * D * 2.0 ** -23 * sden
    worst = np.unravel_index(np.argmax(row_err / row_tol), row_err.shape)
    assert np.all(row_err <= row_tol), (
        f"normalised error {row_err[worst]:.3e} > {row_tol[worst]:.3e} at row {worst}")
    return float(row_err.max())


CASES = {
    # name: (bh, sq, skv, causal, key growth)
    "one_block": (2, 128, 128, False, 0.0),
    "multi_block": (3, 256, 640, False, 0.0),
    "ragged": (2, 200, 333, False, 0.0),
    "tiny": (1, 5, 7, False, 0.0),
    "causal_square": (2, 384, 384, True, 0.0),
    "causal_ragged": (3, 130, 300, True, 0.0),
    "causal_sq_lt_skv": (2, 100, 520, True, 0.0),
    "rising_max": (2, 256, 1024, False, 6.0),
    "rising_max_causal": (2, 512, 512, True, 6.0),
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_attention_parity(dev, case, dt):
    bh, sq, skv, causal, growth = CASES[case]
    seed = bh * 1000 + sq + skv
    q = draw((bh, sq, D), seed, dt)
    k = draw((bh, skv, D), seed + 1, dt)
    v = draw((bh, skv, D), seed + 2, dt)
    if growth:
        # keys grow along the sequence: each block's max moves the reference
        # (the O rescale path)
        ramp = 1.0 + growth * torch.arange(skv, dtype=torch.float32)[None, :, None] / skv
        k = (k.float() * ramp).to(TD[dt])
    scale = 1.0 / math.sqrt(D)
    got = run_attention(dev, q, k, v, bh, sq, skv, scale, causal, dt, runs=2)
    check(got, q, k, v, bh, sq, skv, scale, causal, dt)


def test_attention_large_scale_sharp_softmax(dev):
    """A large scale makes most rows nearly one-hot (the max shift matters)."""
    bh, sq, skv = 2, 256, 384
    q, k, v = draw((bh, sq, D), 5, "bf16"), draw((bh, skv, D), 6, "bf16"), draw((bh, skv, D), 7, "bf16")
    got = run_attention(dev, q, k, v, bh, sq, skv, 0.5, False, "bf16")
    check(got, q, k, v, bh, sq, skv, 0.5, False, "bf16")


def test_attention_constant_values_come_back(dev):
    """V constant along the sequence: every output row is that constant
    (probabilities sum to one), exactly representable."""
    bh, sq, skv = 2, 256, 512
    q, k = draw((bh, sq, D), 8, "bf16"), draw((bh, skv, D), 9, "bf16")
    row = draw((1, 1, D), 10, "bf16")
    v = row.expand(bh, skv, D).contiguous()
    got = run_attention(dev, q, k, v, bh, sq, skv, 0.125, True, "bf16").reshape(bh, sq, D)
    ref = row.float().expand(bh, sq, D)
    assert float((got.float() - ref).abs().max()) <= 2.0 ** -8 * float(ref.abs().max())


def test_attention_empty_and_zero_key_cases(dev):
    # seq_q == 0: nothing is written
    O = torch.full((64,), 3.0, dtype=torch.bfloat16, device=dev)
    plan = H.hgemm_attention_plan_create(2, 0, 16, D, 1.0, 0, DT["bf16"])
    try:
        H.hgemm_attention_run(plan, None, None, None, O)
        assert H.hgemm_attention_check(plan) == 0
    finally:
        H.hgemm_attention_plan_destroy(plan)
    assert torch.all(O.cpu() == 3.0)
    # seq_kv == 0: the empty sum, zeros
    O = torch.full((3 * 10 * D,), 3.0, dtype=torch.float16, device=dev)
    plan = H.hgemm_attention_plan_create(3, 10, 0, D, 1.0, 0, DT["f16"])
    try:
        H.hgemm_attention_run(plan, None, None, None, O)
        assert H.hgemm_attention_check(plan) == 0
    finally:
        H.hgemm_attention_plan_destroy(plan)
    assert torch.all(O.cpu() == 0)


def test_attention_argument_checks(dev):
    with pytest.raises(H.HgemmError) as ei:
        H.hgemm_attention_plan_create(2, 16, 16, 64, 1.0, 0, DT["bf16"])
    assert ei.value.status == 2
    for args in [(2, 32, 16, D, 1.0, 1, DT["bf16"]),    # causal with seq_q > seq_kv
                 (2, 16, 16, D, 0.0, 0, DT["bf16"]),    # scale 0
                 (2, 16, 16, D, float("nan"), 0, DT["bf16"]),
                 (2, 16, 16, D, 1.0, 0, H.HGEMM_F32),   # fp32 inputs
                 (0, 16, 16, D, 1.0, 0, DT["bf16"])]:   # no heads
        with pytest.raises(H.HgemmError) as ei:
            H.hgemm_attention_plan_create(*args)
        assert ei.value.status == 1, args
    plan = H.hgemm_attention_plan_create(1, 16, 16, D, 1.0, 0, DT["bf16"])
    try:
        x = torch.zeros(16 * D + 8, dtype=torch.bfloat16, device=dev)
        with pytest.raises(H.HgemmError) as ei:
            H.hgemm_attention_run(plan, x.data_ptr() + 2, x, x, x)
        assert ei.value.status == 1
    finally:
        H.hgemm_attention_plan_destroy(plan)


def test_attention_host_buffers(dev):
    bh, sq, skv = 2, 192, 320
    q, k, v = draw((bh, sq, D), 11, "f16"), draw((bh, skv, D), 12, "f16"), draw((bh, skv, D), 13, "f16")
    O = torch.empty(bh * sq * D, dtype=torch.float16).pin_memory()
    plan = H.hgemm_attention_plan_create(bh, sq, skv, D, 0.09, 1, DT["f16"])
    try:
        H.hgemm_attention_run_host(plan, q.pin_memory(), k.pin_memory(), v.pin_memory(), O)
        assert H.hgemm_attention_check(plan) == 0
    finally:
        H.hgemm_attention_plan_destroy(plan)
    check(O, q, k, v, bh, sq, skv, 0.09, True, "f16")


@pytest.mark.parametrize("bh,causal", [(24, False), (25, True)])
def test_attention_host_buffers_many_heads(dev, bh, causal):
    """hgemm_attention_run_host on 24 and 25 heads of 1024 x 1024: the last
    query row of every head and random rows match the oracle, and a second
    call gives the same O."""
    sq = skv = 1024
    q, k, v = draw((bh, sq, D), 21, "bf16"), draw((bh, skv, D), 22, "bf16"), draw((bh, skv, D), 23, "bf16")
    O = torch.empty(bh * sq * D, dtype=torch.bfloat16).pin_memory()
    plan = H.hgemm_attention_plan_create(bh, sq, skv, D, 0.0884, int(causal), DT["bf16"])
    try:
        qp, kp, vp = q.pin_memory(), k.pin_memory(), v.pin_memory()
        H.hgemm_attention_run_host(plan, qp, kp, vp, O)
        first = O.clone()
        H.hgemm_attention_run_host(plan, qp, kp, vp, O)
        assert H.hgemm_attention_check(plan) == 0
    finally:
        H.hgemm_attention_plan_destroy(plan)
    assert torch.equal(O, first), "repeated calls differ"
    g = np.random.default_rng(9)
    rb = np.concatenate([np.arange(bh), g.integers(0, bh, 64)])
    ri = np.concatenate([np.full(bh, sq - 1), g.integers(0, sq, 64)])
    check(O, q, k, v, bh, sq, skv, 0.0884, causal, "bf16", rows=(rb, ri))


@pytest.mark.parametrize("causal", [False, True])
def test_attention_full_size_sampled(dev, causal):
    """The attention workload at full size (64 heads x 1024 x 1024, head 128,
    bf16), as the bench runs it, on 192 sampled query rows."""
    from tensor_core_dense_swizzled_gb300 import inputs
    w = inputs.ATTENTION_WORKLOADS["attn_causal" if causal else "attn"]
    q, k, v = inputs.make_attention_inputs(w)
    got = run_attention(dev, q, k, v, w.bh, w.sq, w.skv, w.scale, w.causal, w.dtype)
    g = np.random.default_rng(7)
    rb = g.integers(0, w.bh, 192)
    ri = g.integers(0, w.sq, 192)
    ri[:4] = [0, 1, w.sq - 1, 127]
    check(got, q, k, v, w.bh, w.sq, w.skv, w.scale, w.causal, w.dtype, rows=(rb, ri))
