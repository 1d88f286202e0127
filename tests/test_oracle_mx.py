"""Pins for the oracle's 4-bit (MXFP4) cache format: decode, encoder, block scale and row
quantiser.

The Step-3 page names further KV quantisation as a way to raise MFA's arithmetic intensity
(section 5 "Model-System Co-design", "Quantization and MTP") without fixing a format.  The
cache format taken is the OCP Microscaling (MX) FP4 format: E2M1 elements (1 sign bit, 2
exponent bits with bias 1, 1 mantissa bit, no infinities or NaN) in blocks of 32 consecutive
elements of a token row, each block with one E8M0 scale 2^(e - 127); a block's scale is
2^(floor(log2 amax) - 2) (2 being E2M1's largest exponent), and its elements are rounded to the
nearest E2M1 value of x / scale, ties to the even code, saturating at 6.

What pins it, besides the oracle's own code:
  - torch's float8_e8m0fnu decoder, on all 256 scale codes;
  - the E2M1 value set (the format's table of 8 magnitudes) and exact representability of
    every value in torch's float8_e4m3fn;
  - the input generator's independent numpy quantiser (midpoint search), value by value and
    row by row, and numpy's log2 for the block exponent;
  - torch fp64 SDPA on a numpy dequantisation of an MXFP4 cache;
  - the dequantisation error bound;
  - planted mutants, each of which some pin above rejects.
"""
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle
from decode_attention_02_gb300 import inputs
from test_oracle import assert_close, sdpa_reference

E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e2m1_values(lib=None):
    return np.array([oracle.e2m1_to_double(c, lib=lib) for c in range(16)])


def test_e8m0_every_code_matches_torch():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = np.array([oracle.e8m0_to_double(c) for c in range(256)])
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(got[:255], ref[:255])


def test_e2m1_codes_are_the_format_table():
    v = _e2m1_values()
    assert list(v[:8]) == E2M1_TABLE
    assert list(v[8:]) == [-x for x in E2M1_TABLE]
    # every E2M1 value is an e4m3 value (the kernel decodes E2M1 through e4m3 codes)
    t = torch.tensor(v, dtype=torch.float64)
    assert torch.equal(t.to(torch.float32).to(torch.float8_e4m3fn).to(torch.float64), t)


def _numpy_e2m1(y):
    """The generator's E2M1 rounding of scaled values (midpoint search)."""
    a = np.abs(np.asarray(y, dtype=np.float64))
    lo = np.searchsorted(inputs._E2M1_MID, a, side="left")
    hi = np.searchsorted(inputs._E2M1_MID, a, side="right")
    idx = np.minimum(np.where(lo != hi, lo + (lo % 2), lo), 7)
    return (idx | np.where(np.signbit(y), 8, 0)).astype(np.uint8)


def test_e2m1_encoder_rounds_to_nearest_even_and_saturates():
    mids = list(inputs._E2M1_MID)
    probe = [0.0, -0.0, 6.0, 6.5, 1e9, -1e9, 1e-30, -1e-30] + E2M1_TABLE
    for m in mids:
        probe += [m, np.nextafter(m, 0.0), np.nextafter(m, 10.0)]
    rng = np.random.default_rng(5)
    probe += list(rng.uniform(-8, 8, size=2000))
    probe = np.array(probe + [-x for x in probe])
    got = np.array([oracle.e2m1_from_double(float(x)) for x in probe], dtype=np.uint8)
    assert np.array_equal(got, _numpy_e2m1(probe))
    # ties: 0.25 -> 0, 0.75 -> 1.0, 1.25 -> 1.0, 1.75 -> 2.0, 2.5 -> 2.0, 3.5 -> 4.0, 5 -> 4.0
    assert [oracle.e2m1_from_double(m) for m in mids] == [0, 2, 2, 4, 4, 6, 6]
    assert oracle.e2m1_from_double(-0.1) == 8   # a negative value rounding to zero keeps its sign


def test_mx_block_exponent_is_floor_log2_amax_minus_2():
    rng = np.random.default_rng(6)
    cases = [np.zeros(32, np.float32), np.full(32, 6.0, np.float32), np.full(32, 7.0, np.float32),
             np.full(32, 2.0 ** -130, np.float32), np.full(32, 3.0e38, np.float32)]
    cases += [(rng.standard_normal(32) * 2.0 ** rng.integers(-40, 40)).astype(np.float32) for _ in range(200)]
    for x in cases:
        amax = float(np.abs(x).max())
        want = -127 if amax == 0 else int(np.clip(np.floor(np.log2(np.float64(amax))) - 2, -127, 127))
        assert oracle.mx_block_exponent(x) == want, (amax, want)


def _rows(n, d=256, seed=7):
    return inputs.new_token_rows(n, d, seed=seed)


def test_mx_row_quantiser_matches_the_generator():
    """The oracle's append into an MXFP4 cache writes the codes and scales the generator's
    numpy quantiser gives for the same bf16 rows (all eight row kinds)."""
    n = 64
    k_new, v_new = _rows(n, seed=8), _rows(n, seed=9)
    case = inputs.small("mxq", n, [1] * n, kv_dtype="mxfp4", seed=10, extra_blocks=0)
    pos = torch.zeros(n, dtype=torch.int32)
    kc, vc, ks, vs, mask = oracle.kv_append(k_new, v_new, pos, case.block_table, case.k_cache, case.v_cache,
                                            case.k_scale, case.v_scale)
    assert mask == 0
    table = case.block_table.numpy()[:, 0]
    for new, cache, sc in ((k_new, kc, ks), (v_new, vc, vs)):
        want_c, want_s = inputs._to_mxfp4(new.float().numpy())
        assert np.array_equal(cache[table, 0], want_c.numpy())
        assert np.array_equal(sc[table, 0], want_s.numpy())


def test_mx_dequantisation_error_bound():
    """|x - dequant(quant(x))| is at most half a code step of its block, except where |x| is
    above 6 scales (saturated at 6 scales)."""
    n = 48
    x = _rows(n, seed=11)
    case = inputs.small("mxb", n, [1] * n, kv_dtype="mxfp4", seed=12, extra_blocks=0)
    kc, vc, ks, vs, mask = oracle.kv_append(x, x, torch.zeros(n, dtype=torch.int32), case.block_table,
                                            case.k_cache, case.v_cache, case.k_scale, case.v_scale)
    table = case.block_table.numpy()[:, 0]
    codes, scales = kc[table, 0], ks[table, 0]
    vals = _e2m1_values()
    full = np.empty((n, 256), dtype=np.uint8)
    full[:, 0::2], full[:, 1::2] = codes & 15, codes >> 4
    sc = np.repeat(np.ldexp(1.0, scales.astype(int) - 127), 32, axis=1)
    deq = vals[full] * sc
    xf = x.float().numpy().astype(np.float64)
    step = np.where(np.abs(deq) < 2 * sc, 0.5 * sc, np.where(np.abs(deq) < 4 * sc, sc, 2 * sc))
    err = np.abs(xf - deq)
    sat = np.abs(xf) > 6 * sc
    assert np.all((err <= step / 2 + 1e-300) | sat)
    assert np.all(np.abs(deq[sat]) == 6 * sc[sat])


@pytest.mark.parametrize("kw", [dict(), dict(head_dim=128, num_kv_heads=4), dict(head_dim=512, num_q_heads=16, kv_shared=True)])
def test_mxfp4_decode_matches_sdpa_on_a_numpy_dequantisation(kw):
    """The dense gather of the SDPA reference decodes MXFP4 rows with the format's value table
    and torch's E8M0 decoder; here the whole decode is checked, for the grouped and shared
    shapes too."""
    case = inputs.small("mxd", 3, [1, 70, 200], kv_dtype="mxfp4", seed=13, **kw)
    out, lse = oracle.decode(case)
    ro, rl = sdpa_reference(case)
    assert_close(out, ro)
    assert_close(lse, rl)


# ------------------------------------------------------------- mutation check

_MUTANTS = {
    "mx_nibble_order": ("(e & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15)",
                        "(e & 1) ? (uint8_t)(byte & 15) : (uint8_t)(byte >> 4)"),
    "mx_scale_block": ("+ e / 32])", "+ e / 64])"),
    "e8m0_bias": ("ldexp(1.0, (int)e - 127)", "ldexp(1.0, (int)e - 126)"),
    "e2m1_subnormal": ("(double)m / 2.0 : ldexp", "(double)m / 4.0 : ldexp"),
    "e2m1_bias": ("ldexp(1.0 + (double)m / 2.0, e - 1)", "ldexp(1.0 + (double)m / 2.0, e)"),
    "e2m1_ties_odd": ("e2m1_to_double((uint8_t)c) - a);\n            if (dist < bd || (dist == bd && (c & 1) == 0))",
                      "e2m1_to_double((uint8_t)c) - a);\n            if (dist < bd || (dist == bd && (c & 1) == 1))"),
    "e2m1_no_saturation": ("    int best = 7;\n    if (a < 6.0) {", "    int best = 0;\n    if (a < 6.0) {"),
    "mx_exponent_off_by_one": ("int e = (E - 1) - 2;", "int e = (E - 1) - 1;"),
    "mx_codes_unscaled": ("ldexp((double)blk[i], -e)", "(double)blk[i]"),
}


def _pins_pass(lib):
    try:
        v = _e2m1_values(lib)
        if list(v[:8]) != E2M1_TABLE or list(v[8:]) != [-x for x in E2M1_TABLE]:
            return False
        ref = torch.arange(255, dtype=torch.int32).to(torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
        if not np.array_equal([oracle.e8m0_to_double(c, lib=lib) for c in range(255)], ref):
            return False
        probe = np.concatenate([inputs._E2M1_MID, np.linspace(-7, 7, 281)])
        if not np.array_equal([oracle.e2m1_from_double(float(x), lib=lib) for x in probe], _numpy_e2m1(probe)):
            return False
        x = (np.random.default_rng(14).standard_normal(32) * 3).astype(np.float32)
        if oracle.mx_block_exponent(x, lib=lib) != int(np.floor(np.log2(np.abs(x).max())) - 2):
            return False
        n = 16
        k_new = _rows(n, seed=15)
        case = inputs.small("mxm", n, [1] * n, kv_dtype="mxfp4", seed=16, extra_blocks=0)
        kc, vc, ks, vs, mask = oracle.kv_append(k_new, k_new, torch.zeros(n, dtype=torch.int32), case.block_table,
                                                case.k_cache, case.v_cache, case.k_scale, case.v_scale, lib=lib)
        want_c, want_s = inputs._to_mxfp4(k_new.float().numpy())
        table = case.block_table.numpy()[:, 0]
        if not (np.array_equal(kc[table, 0], want_c.numpy()) and np.array_equal(ks[table, 0], want_s.numpy())):
            return False
        dcase = inputs.small("mxm2", 2, [70, 131], kv_dtype="mxfp4", seed=17)
        out, lse = oracle.decode(dcase, lib=lib)
        ro, rl = sdpa_reference(dcase)
        assert_close(out, ro)
        assert_close(lse, rl)
    except AssertionError:
        return False
    return True


def test_mx_mutants_are_caught():
    src = open(os.path.join(os.path.dirname(oracle.__file__), "mfa_oracle.c")).read()
    assert _pins_pass(oracle._load())
    with tempfile.TemporaryDirectory() as tmp:
        for name, (old, new) in _MUTANTS.items():
            assert src.count(old) == 1, f"mutant {name}: pattern found {src.count(old)} times"
            path = os.path.join(tmp, f"{name}.c")
            with open(path, "w") as f:
                f.write(src.replace(old, new))
            so = os.path.join(tmp, f"{name}.so")
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                                   "-fno-fast-math", "-ffp-contract=off", "-o", so, path, "-lm"])
            assert not _pins_pass(oracle.load_library(so)), f"mutant {name} survived the pins"
