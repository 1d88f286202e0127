"""Parity of the e4m3-KV path with the fp64 oracle fed the same dequantised values.

Limits for FP8 KV: max-abs <= 3e-2 and relative-L2 <= 1.5e-2 (on the fp32 result;
the bf16 output may add half a bf16 ulp).  The oracle decodes every e4m3 code
exactly and multiplies by its per-token scale in double precision.
"""
import numpy as np
import pytest
import torch

import decode_attention_02_gb300 as mfa
import oracle
from decode_attention_02_gb300 import inputs
from test_gpu_parity import check_parity, gpu_decode, to_dev

pytestmark = pytest.mark.gpu

FP8 = dict(max_abs=3e-2, rel_l2=1.5e-2)


def test_fp8_length_one_returns_the_dequantised_value():
    # one token: the output is v_0 (code * scale); exercises the V-scale folding alone
    case = inputs.small("f1", 3, [1, 1, 1], kv_dtype="fp8_e4m3", seed=40)
    out, lse, _ = gpu_decode(case)
    check_parity(case, out, lse, **FP8)


def test_fp8_two_tokens():
    case = inputs.small("f2", 3, [2, 2, 2], kv_dtype="fp8_e4m3", seed=41)
    out, lse, _ = gpu_decode(case)
    check_parity(case, out, lse, **FP8)


@pytest.mark.parametrize("force_ctas", [0, 1, 3, 16, 64])
def test_fp8_ragged_lengths_any_split(force_ctas):
    lens = [1, 63, 64, 65, 127, 128, 129, 200, 0, 517, 1000, 300]
    case = inputs.small("fr", len(lens), lens, kv_dtype="fp8_e4m3", seed=42, extra_blocks=3)
    out, lse, _ = gpu_decode(case, force_ctas=force_ctas)
    check_parity(case, out, lse, **FP8)


def test_fp8_bf16_output_is_rne_of_fp32_output():
    case = inputs.small("fo", 4, [3000, 1, 700, 1500], kv_dtype="fp8_e4m3", seed=43)
    o32, l32, _ = gpu_decode(case, force_ctas=5)
    o16, l16, _ = gpu_decode(case, force_ctas=5, out_dtype=mfa.MFA_OUT_BF16)
    assert torch.equal(o16.view(torch.int16), o32.to(torch.bfloat16).view(torch.int16))
    ref = oracle.decode(case)
    check_parity(case, o32, l32, ref=ref, **FP8)
    check_parity(case, o16, l16, ref=ref, **FP8)


@pytest.mark.parametrize("force_ctas", [0, 5])
def test_fp8_v_scales_over_a_wide_range(force_ctas):
    """Per-token V scales from about 2^-26 to 2^8 (V rows of absmax from about 1e-6 to 5e4):
    sequence b's V rows are scaled by 2^base[b] and each token further by 2^U[-3, 3].  The
    output of sequence b scales with it, so the FP8 bar applies to out / (2^base[b] * 2^3).
    No device status bit may be set (the check flag raises on one)."""
    lens = [700, 1500, 64, 300, 2000, 129, 1000, 450]
    base = [-16, -12, -8, -4, 0, 4, 8, 12]
    case = inputs.small("fvr", len(lens), lens, kv_dtype="fp8_e4m3", seed=44)
    rng = np.random.default_rng(44)
    vs = case.v_scale.numpy()
    table = case.block_table.numpy()
    for b, L in enumerate(lens):
        t = np.arange(L)
        mult = np.exp2(base[b] + rng.integers(-3, 4, size=L)).astype(np.float32)
        vs[table[b, t // 64], t % 64] *= mult
    assert vs[np.isfinite(vs)].min() < 2.0 ** -24 and vs[np.isfinite(vs)].max() > 2.0 ** 7
    out, lse, _ = gpu_decode(case, force_ctas=force_ctas)
    ref_o, ref_lse = oracle.decode(case)
    got = out.double().cpu().numpy()
    for b in range(len(lens)):
        f = 2.0 ** (base[b] + 3)
        g, r = got[b] / f, ref_o[b] / f
        assert np.abs(g - r).max() <= FP8["max_abs"], f"sequence {b}: max-abs {np.abs(g - r).max():.3e}"
        rel = np.linalg.norm(g - r) / np.linalg.norm(r)
        assert rel <= FP8["rel_l2"], f"sequence {b}: rel-L2 {rel:.3e}"
    assert np.abs(lse.double().cpu().numpy() - ref_lse).max() <= 2e-3


def test_fp8_q_beyond_the_f16_range():
    # q.K^T runs on e4m3 codes with q split into hi + lo under a per-sequence power of two,
    # so a q far outside the f16 range is still exact (here: one-hot attention)
    case = inputs.small("fq", 3, [300, 129, 64], kv_dtype="fp8_e4m3", seed=45)
    case.q[0] *= 2.0 ** 20
    case.q[2] *= 2.0 ** -20
    out, lse, _ = gpu_decode(case)
    ref_o, ref_lse = oracle.decode(case)
    got = out.double().cpu().numpy()
    assert np.abs(got - ref_o).max() <= FP8["max_abs"]
    assert np.linalg.norm(got - ref_o) / np.linalg.norm(ref_o) <= FP8["rel_l2"]
    # lse of sequence 0 is ~3e6: the fp32 scores that make it carry the accumulator's
    # relative rounding (about 1e-6 over 256 products), so the bound is relative there
    g = lse.double().cpu().numpy()
    assert np.all(np.abs(g - ref_lse) <= 2e-3 + 1e-5 * np.abs(ref_lse))


def test_fp8_heads_of_mixed_magnitude_share_one_split_scale():
    case = inputs.small("fm", 2, [700, 1500], kv_dtype="fp8_e4m3", seed=46)
    mult = torch.tensor([2.0 ** ((h % 9) - 4) for h in range(64)], dtype=torch.float32)
    case.q.copy_((case.q.float() * mult[None, :, None]).to(torch.bfloat16))
    out, lse, _ = gpu_decode(case, force_ctas=3)
    check_parity(case, out, lse, **FP8)


@pytest.mark.parametrize("name", ["b128_l4096_fp8", "b32_l4096_fp8", "long_b4_l131072_fp8"])
def test_fp8_full_size_workload(name):
    case = inputs.generate(inputs.WORKLOADS[name])
    out, lse, dec = gpu_decode(case)
    assert dec.plan.num_ctas == min(torch.cuda.get_device_properties(0).multi_processor_count,
                                    int(dec.plan.total_tiles))
    check_parity(case, out, lse, **FP8)


def test_fp8_ragged_full_size_mix():
    """128 sequences of 1,024..8,192 tokens in e4m3 (ragged last pages, 1% of K elements x20):
    many sequence switches per CTA under the e4m3 schedule's boundary weight."""
    import dataclasses
    w = dataclasses.replace(inputs.WORKLOADS["ragged_b128_l1024_8192_bf16"], name="ragged_b128_l1024_8192_fp8",
                            kv_dtype="fp8_e4m3", seed=12)
    case = inputs.generate(w)
    out, lse, dec = gpu_decode(case)
    assert dec.plan.num_ctas == torch.cuda.get_device_properties(0).multi_processor_count
    check_parity(case, out, lse, **FP8)
