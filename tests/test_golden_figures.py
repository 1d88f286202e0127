"""The workload shape and the per-token work formulas against the figures the
Step-3 page prints (section 5 "Model-System Co-design", "Attention Design").

The page gives MFA's arithmetic intensity with 8-bit KV (128 FLOPs per byte),
its effective rank (16,384) and, for DeepSeek-V3's MLA, intensity 512 and a
compute ratio of 1/4.  Counting a multiply-add as two FLOPs, decode attention
with one shared K head and one shared V head does 4*H*d FLOPs per cached token
and, at 8 bits, reads 2*d bytes of it, so the intensity is 2*H: the printed 128
fixes H = 64 and the rank H*d = 16,384 fixes d = 256.  The MLA figures (128
heads over a 512-wide latent that serves as both K and V) check the same
counting convention.  bench.py's byte and FLOP formulas must reproduce these.
"""
import os

import pytest

import bench
from decode_attention_02_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "step3_mfa_printed_figures.txt")


def _figures():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if len(line) >= 2:
                vals[line[0]] = float(line[1])
    return vals


def test_fixture_holds_every_figure():
    assert set(_figures()) == {"mfa_intensity_8bit_kv", "mla_dsv3_intensity_8bit_kv", "mfa_effective_rank",
                               "mla_dsv3_effective_rank", "gqa_qwen3_effective_rank", "mfa_over_dsv3_compute"}


def test_printed_intensity_and_rank_fix_the_shape():
    g = _figures()
    H = g["mfa_intensity_8bit_kv"] / 2          # 4Hd FLOPs / 2d bytes = 2H
    d = g["mfa_effective_rank"] / H
    assert (H, d) == (inputs.NUM_Q_HEADS, inputs.HEAD_DIM) == (64, 256)
    # Qwen3's printed rank is 64 heads of width 128 under the same product
    assert g["gqa_qwen3_effective_rank"] == 64 * 128


def test_flop_formula_gives_the_printed_intensity():
    g = _figures()
    H, d = inputs.NUM_Q_HEADS, inputs.HEAD_DIM
    flops_per_token = bench.algorithmic_flops([1], H, d)
    kv_bytes_8bit = 2 * d                        # one K row and one V row of d bytes
    assert flops_per_token / kv_bytes_8bit == g["mfa_intensity_8bit_kv"]
    assert bench.intensity_per_token("fp8_e4m3", H, d, kv_heads_bytes=kv_bytes_8bit) == g["mfa_intensity_8bit_kv"]
    # the stored per-token scales (two fp32) lower it slightly: 65,536 / 520
    assert bench.intensity_per_token("fp8_e4m3", H, d) == pytest.approx(65536 / 520)
    assert bench.intensity_per_token("bf16", H, d) == g["mfa_intensity_8bit_kv"] / 2


def test_same_convention_reproduces_the_mla_figures():
    g = _figures()
    H_mla, latent = 128, 512                     # 128 heads over one shared 512-wide latent (K = V)
    flops = bench.algorithmic_flops([1], H_mla, latent)
    assert flops / latent == g["mla_dsv3_intensity_8bit_kv"]
    assert bench.algorithmic_flops([1], 64, 256) / flops == g["mfa_over_dsv3_compute"]


def test_byte_formula_per_token_and_per_sequence():
    lens = [4096, 1, 0, 65]
    for dt, per_tok in (("bf16", 1024), ("fp8_e4m3", 520)):
        a = bench.algorithmic_bytes(lens, dt)
        assert a["kv"] == sum(lens) * per_tok
        pages = 64 + 1 + 0 + 2
        assert a["total"] - a["kv"] == 4 * (2 * 64 * 256 * 2 + 4 + 64 * 4) + pages * 4
