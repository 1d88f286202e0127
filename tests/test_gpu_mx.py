"""Parity of the MXFP4-KV path (OCP MX FP4: E2M1 codes, one E8M0 scale per 32 elements of a
row) with the fp64 oracle fed the same dequantised values.

The kernel converts each 4-bit row on chip to e4m3 codes under one power-of-two scale per row
(exact for every block whose scale is at least 2^-14 of the row's largest) and from there runs
the e4m3 path, so the e4m3 path's limits apply: max-abs <= 3e-2 and relative-L2 <= 1.5e-2 on
the fp32 result, lse to 2e-3.
"""
import dataclasses

import numpy as np
import pytest
import torch

import decode_attention_02_gb300 as mfa
import oracle
from decode_attention_02_gb300 import inputs
from test_gpu_parity import check_parity, gpu_decode

pytestmark = pytest.mark.gpu

MX = dict(max_abs=3e-2, rel_l2=1.5e-2)


def _used_rows(case):
    """(page, slot) of every cached token of every sequence: [(b, blocks, slots)]."""
    table = case.block_table.numpy()
    out = []
    for b, L in enumerate(case.seq_lens.tolist()):
        t = np.arange(L)
        out.append((b, table[b, t // 64], t % 64))
    return out


def test_mx_length_one_returns_the_dequantised_value():
    case = inputs.small("m1", 3, [1, 1, 1], kv_dtype="mxfp4", seed=140)
    out, lse, _ = gpu_decode(case)
    check_parity(case, out, lse, **MX)


def test_mx_two_tokens():
    case = inputs.small("m2", 3, [2, 2, 2], kv_dtype="mxfp4", seed=141)
    out, lse, _ = gpu_decode(case)
    check_parity(case, out, lse, **MX)


@pytest.mark.parametrize("force_ctas", [0, 1, 3, 16, 64])
def test_mx_ragged_lengths_any_split(force_ctas):
    lens = [1, 63, 64, 65, 127, 128, 129, 200, 0, 517, 1000, 300]
    case = inputs.small("mr", len(lens), lens, kv_dtype="mxfp4", seed=142, extra_blocks=3)
    out, lse, _ = gpu_decode(case, force_ctas=force_ctas)
    check_parity(case, out, lse, **MX)


def test_mx_bf16_output_is_rne_of_fp32_output():
    case = inputs.small("mo", 4, [3000, 1, 700, 1500], kv_dtype="mxfp4", seed=143)
    o32, l32, _ = gpu_decode(case, force_ctas=5)
    o16, l16, _ = gpu_decode(case, force_ctas=5, out_dtype=mfa.MFA_OUT_BF16)
    assert torch.equal(o16.view(torch.int16), o32.to(torch.bfloat16).view(torch.int16))
    ref = oracle.decode(case)
    check_parity(case, o32, l32, ref=ref, **MX)
    check_parity(case, o16, l16, ref=ref, **MX)


@pytest.mark.parametrize("force_ctas", [0, 5])
def test_mx_block_scales_over_a_wide_range(force_ctas):
    """Within a row, block scales up to 2^-24 below the row's largest (every block of K and V
    lowered by U[0, 24] binades: the table-shift, rounded-table and subnormal-grid conversions
    all run); across sequences, V scaled by 2^base[b] with base from -40 to 40 (the output of
    sequence b scales with it, so the bar applies to out / 2^base[b])."""
    lens = [700, 1500, 64, 300, 2000, 129, 1000, 450]
    base = [-40, -24, -8, 0, 8, 16, 24, 40]
    case = inputs.small("mw", len(lens), lens, kv_dtype="mxfp4", seed=144)
    rng = np.random.default_rng(144)
    ks, vs = case.k_scale.numpy(), case.v_scale.numpy()
    for b, blks, slots in _used_rows(case):
        n = len(blks)
        ks[blks, slots] = np.clip(ks[blks, slots].astype(int) - rng.integers(0, 25, size=(n, 8)), 1, 254)
        vs[blks, slots] = np.clip(vs[blks, slots].astype(int) + base[b] - rng.integers(0, 25, size=(n, 8)), 1, 254)
    out, lse, _ = gpu_decode(case, force_ctas=force_ctas)
    ref_o, ref_lse = oracle.decode(case)
    got = out.double().cpu().numpy()
    for b in range(len(lens)):
        f = 2.0 ** base[b]
        g, r = got[b] / f, ref_o[b] / f
        assert np.abs(g - r).max() <= MX["max_abs"], f"sequence {b}: max-abs {np.abs(g - r).max():.3e}"
        rel = np.linalg.norm(g - r) / np.linalg.norm(r)
        assert rel <= MX["rel_l2"], f"sequence {b}: rel-L2 {rel:.3e}"
    assert np.abs(lse.double().cpu().numpy() - ref_lse).max() <= 2e-3


def test_mx_tiny_scales_use_the_smallest_row_scale():
    """Rows whose largest scale byte is below 7 take the row scale 2^-126 (the reference
    exponent's floor): V scale bytes 0..6 in sequence 0, K scale bytes 0..6 in sequence 1."""
    lens = [300, 200, 129]
    case = inputs.small("mt", len(lens), lens, kv_dtype="mxfp4", seed=145)
    rng = np.random.default_rng(145)
    rows = _used_rows(case)
    b, blks, slots = rows[0]
    case.v_scale.numpy()[blks, slots] = rng.integers(0, 7, size=(len(blks), 8))
    b, blks, slots = rows[1]
    case.k_scale.numpy()[blks, slots] = rng.integers(0, 7, size=(len(blks), 8))
    out, lse, _ = gpu_decode(case)
    ref_o, ref_lse = oracle.decode(case)
    got = out.double().cpu().numpy()
    f0 = 2.0 ** (6 - 127 + 3)
    assert np.abs(got[0] / f0 - ref_o[0] / f0).max() <= MX["max_abs"]
    assert np.abs(got[1:] - ref_o[1:]).max() <= MX["max_abs"]
    assert np.abs(lse.double().cpu().numpy() - ref_lse).max() <= 2e-3


@pytest.mark.parametrize("T", [2, 4])
def test_mx_multi_token_decode(T):
    lens = [1, 2, 64, 65, 130, 700, 3, 0]
    case = inputs.small("mm", len(lens), lens, kv_dtype="mxfp4", seed=147 + T, tokens_per_seq=T)
    out, lse, _ = gpu_decode(case, force_ctas=7)
    check_parity(case, out, lse, **MX)


@pytest.mark.parametrize("name", ["b128_l4096_mxfp4", "b32_l4096_mxfp4"])
def test_mx_full_size_workload(name):
    case = inputs.generate(inputs.WORKLOADS[name])
    out, lse, dec = gpu_decode(case)
    assert dec.plan.num_ctas == min(torch.cuda.get_device_properties(0).multi_processor_count,
                                    int(dec.plan.total_tiles))
    check_parity(case, out, lse, **MX)


def test_mx_ragged_full_size_mix():
    """128 sequences of 1,024..8,192 tokens in MXFP4 (ragged last pages, 1% of K elements x20)."""
    w = dataclasses.replace(inputs.WORKLOADS["ragged_b128_l1024_8192_bf16"], name="ragged_b128_l1024_8192_mxfp4",
                            kv_dtype="mxfp4", seed=13)
    case = inputs.generate(w)
    out, lse, dec = gpu_decode(case)
    assert dec.plan.num_ctas == torch.cuda.get_device_properties(0).multi_processor_count
    check_parity(case, out, lse, **MX)
