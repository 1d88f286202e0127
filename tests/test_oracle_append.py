"""Pins for the oracle's KV append (new key/value rows into the paged cache, FP8 quantised).

The attention instances own and fill their KV caches (Step-3, paperlayer.ai/abs/2507.19427v1,
section 7 "Implementation and Results"), which hold 8-bit KV (section 5 "Model-System
Co-design").  The e4m3 format and its round-to-nearest-even rule come from the OCP FP8
definition; the per-row scale absmax/448 is the storage format the decode reads.  The pins:
torch's float8_e4m3fn cast (a library encoder) on every fp32 value where a rounding rule
could go wrong, round trips of every code, saturation and signed zeros, the input
generator's own numpy/torch quantiser on whole rows, the dequantisation error bound, and
slots other than the target left unchanged.  ``test_append_mutants_are_caught`` plants
mistakes in copies of the oracle and checks that these pins reject each one.
"""
import os
import subprocess
import tempfile

import numpy as np
import torch

import oracle
from decode_attention_02_gb300 import inputs

E4M3_MAX = 448.0


def e4m3_values():
    """Values of the non-negative finite codes 0x00..0x7E, by torch's decoder."""
    codes = torch.arange(0x7F, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_e4m3(y: np.ndarray) -> np.ndarray:
    """torch's fp32 -> e4m3 cast (round to nearest even), for |y| <= 448."""
    return torch.from_numpy(np.ascontiguousarray(y, dtype=np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def encoder_probe_values():
    """fp32 values where an e4m3 rounding rule can go wrong, plus random ones."""
    v = e4m3_values()
    mids = ((v[:-1] + v[1:]) / 2).astype(np.float32)   # exact in fp32
    up = np.nextafter(mids, np.float32(np.inf))
    down = np.nextafter(mids, np.float32(-np.inf))
    rng = np.random.default_rng(11)
    uni = rng.uniform(-E4M3_MAX, E4M3_MAX, 50000).astype(np.float32)
    logu = (np.exp2(rng.uniform(-14, np.log2(E4M3_MAX), 50000)) *
            np.where(rng.random(50000) < 0.5, -1, 1)).astype(np.float32)
    pos = np.concatenate([v.astype(np.float32), mids, up, down])
    return np.concatenate([pos, -pos, uni, logu, np.float32([E4M3_MAX, -E4M3_MAX])])


def check_encoder(lib=None):
    y = encoder_probe_values()
    y = y[np.abs(y) <= E4M3_MAX]
    got = oracle.e4m3_from_float_array(y, lib=lib)
    ref = torch_e4m3(y)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} codes differ from torch"


def check_round_trip(lib=None):
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = oracle.e4m3_from_float_array(vals, lib=lib)
    assert np.array_equal(got, codes)


def check_saturation_and_zeros(lib=None):
    # (a list: 0.0 and -0.0 would be one dict key)
    cases = [(448.0, 0x7E), (449.0, 0x7E), (464.0, 0x7E), (479.9, 0x7E), (480.0, 0x7E), (1e30, 0x7E),
             (float("inf"), 0x7E), (-448.0, 0xFE), (-1e30, 0xFE), (float("-inf"), 0xFE),
             (0.0, 0x00), (-0.0, 0x80), (2.0 ** -10, 0x00), (-(2.0 ** -10), 0x80),
             (2.0 ** -9, 0x01), (3 * 2.0 ** -11, 0x01), (2.0 ** -11, 0x00), (-1e-30, 0x80)]
    y = np.array([c[0] for c in cases], dtype=np.float32)
    got = oracle.e4m3_from_float_array(y, lib=lib)
    want = np.array([c[1] for c in cases], dtype=np.uint8)
    assert np.array_equal(got, want), list(zip(y, got, want))


def _append_case(kv_dtype, seed):
    lens = [1, 64, 65, 127, 128, 129, 200, 7, 300, 63, 2, 192, 256, 5, 66, 190, 33]
    case = inputs.small("append", len(lens), lens, kv_dtype=kv_dtype, seed=seed)
    step = inputs.append_step(case, seed=seed + 1, inactive_every=5)
    return case, step


def _changed_rows(before, after):
    """(block, slot) pairs whose row differs (NaN-aware for float arrays)."""
    b = before.reshape(before.shape[0], before.shape[1], -1)
    a = after.reshape(after.shape[0], after.shape[1], -1)
    if np.issubdtype(b.dtype, np.floating):
        diff = ~((a == b) | (np.isnan(a) & np.isnan(b)))
    else:
        diff = a != b
    return set(map(tuple, np.argwhere(diff.any(axis=-1))))


def _targets(case, step):
    table = case.block_table.numpy()
    out = {}
    for b, t in enumerate(step.positions.tolist()):
        if t >= 0:
            out[b] = (int(table[b, t // 64]), t % 64)
    return out


def check_bf16_append(lib=None):
    case, step = _append_case("bf16", 41)
    kc0 = case.k_cache.view(torch.int16).numpy()
    vc0 = case.v_cache.view(torch.int16).numpy()
    kc, vc, _, _, mask = oracle.kv_append(step.k_new, step.v_new, step.positions, case.block_table,
                                          case.k_cache, case.v_cache, lib=lib)
    assert mask == 0
    tg = _targets(case, step)
    kn = step.k_new.view(torch.int16).numpy()
    vn = step.v_new.view(torch.int16).numpy()
    for b, (blk, slot) in tg.items():
        assert np.array_equal(kc[blk, slot], kn[b]) and np.array_equal(vc[blk, slot], vn[b])
    want = set(tg.values())
    # a target slot may already hold the row bits (an all-zero row over old zeros): subset
    assert _changed_rows(kc0, kc) <= want and _changed_rows(vc0, vc) <= want
    assert len(_changed_rows(kc0, kc)) >= len(want) - 4


def _dequant(codes, scale):
    v = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return v * np.float64(scale)


def check_fp8_append(lib=None):
    case, step = _append_case("fp8_e4m3", 43)
    kc, vc, ks, vs, mask = oracle.kv_append(step.k_new, step.v_new, step.positions, case.block_table,
                                            case.k_cache, case.v_cache, case.k_scale, case.v_scale, lib=lib)
    assert mask == 0
    tg = _targets(case, step)
    for rows, cache, scales, name in ((step.k_new, kc, ks, "k"), (step.v_new, vc, vs, "v")):
        x32 = rows.to(torch.float32).numpy()
        # the input generator's own quantiser (numpy division, torch cast) on the same values
        gen_codes, gen_scale = inputs._to_e4m3(x32)
        gen_codes, gen_scale = gen_codes.numpy(), gen_scale.numpy()
        for b, (blk, slot) in tg.items():
            c, s, x = cache[blk, slot], scales[blk, slot], x32[b]
            assert np.array_equal(c, gen_codes[b]), (name, b)
            assert s.view(np.uint32) == gen_scale[b].view(np.uint32), (name, b)
            absmax = np.abs(x).max()
            if absmax == 0:
                assert s == np.float32(1.0) and np.all((c & 0x7F) == 0)
                assert np.array_equal(c == 0x80, np.signbit(x))
                continue
            # the row maximum lands on the largest code, with its sign
            i = int(np.argmax(np.abs(x)))
            assert (c[i] & 0x7F) == 0x7E and bool(c[i] & 0x80) == bool(x[i] < 0)
            # dequantisation error: half an e4m3 step (2^-4 relative in the normal range,
            # 2^-10 in units of the scale below 2^-6), plus the two fp32 roundings
            err = np.abs(_dequant(c, s) - x.astype(np.float64))
            bound = 2.0 ** -4 * np.abs(x) + 2.0 ** -10 * float(s) + 1e-6 * np.abs(x)
            assert np.all(err <= bound), (name, b, float((err - bound).max()))
            # the scale is within a rounding of absmax / 448
            assert abs(float(s) * E4M3_MAX - float(absmax)) <= 2.0 ** -23 * float(absmax)
    want = set(tg.values())
    for before, after in ((case.k_cache.numpy(), kc), (case.v_cache.numpy(), vc),
                          (case.k_scale.numpy()[..., None], ks[..., None]),
                          (case.v_scale.numpy()[..., None], vs[..., None])):
        assert _changed_rows(before, after) <= want


def check_error_masks(lib=None):
    case, step = _append_case("fp8_e4m3", 47)
    pos = step.positions.clone()
    table = case.block_table.clone()
    pos[0] = 64 * table.shape[1]            # beyond the table: reported, skipped
    b_bad = 2
    t = int(pos[b_bad])
    table[b_bad, t // 64] = case.k_cache.shape[0]   # page id outside the pool
    kc, vc, ks, vs, mask = oracle.kv_append(step.k_new, step.v_new, pos, table, case.k_cache, case.v_cache,
                                            case.k_scale, case.v_scale, lib=lib)
    assert mask == oracle.APPEND_BAD_BLOCK | oracle.APPEND_BAD_POSITION
    good = {b: v for b, v in _targets(case, step).items() if b not in (0, b_bad)}
    assert _changed_rows(case.k_cache.numpy(), kc) <= set(good.values())
    # no new tokens at all: nothing changes
    none = torch.full_like(pos, -1)
    kc2, _, ks2, _, mask2 = oracle.kv_append(step.k_new, step.v_new, none, case.block_table, case.k_cache,
                                             case.v_cache, case.k_scale, case.v_scale, lib=lib)
    assert mask2 == 0 and np.array_equal(kc2, case.k_cache.numpy())
    assert np.array_equal(ks2.view(np.uint32), case.k_scale.numpy().view(np.uint32))


def check_multi_token_append(lib=None):
    """T new rows per sequence land at positions[b] .. positions[b] + T - 1: the same bytes
    as T single-row appends at those positions (the single-row append is pinned above)."""
    for kv in ("bf16", "fp8_e4m3"):
        T = 3
        case = inputs.small("append_t", 6, [3, 64, 66, 130, 2, 200], kv_dtype=kv, seed=91, tokens_per_seq=T)
        step = inputs.append_step(case, seed=92, tokens_per_seq=T)
        many = oracle.kv_append(step.k_new, step.v_new, step.positions, case.block_table, case.k_cache,
                                case.v_cache, case.k_scale, case.v_scale, tokens_per_seq=T, lib=lib)
        kc, vc, ks, vs = case.k_cache, case.v_cache, case.k_scale, case.v_scale
        for i in range(T):
            pos_i = torch.where(step.positions >= 0, step.positions + i, step.positions)
            kc, vc, ks, vs, mask = oracle.kv_append(step.k_new[i::T].contiguous(), step.v_new[i::T].contiguous(),
                                                    pos_i, case.block_table, kc, vc, ks, vs, lib=lib)
            kc, vc = torch.from_numpy(kc).view(case.k_cache.dtype), torch.from_numpy(vc).view(case.v_cache.dtype)
            if ks is not None:
                ks, vs = torch.from_numpy(ks), torch.from_numpy(vs)
            assert mask == 0
        assert many[4] == 0
        assert np.array_equal(many[0], kc.view(torch.uint8 if kv != "bf16" else torch.int16).numpy())
        assert np.array_equal(many[1], vc.view(torch.uint8 if kv != "bf16" else torch.int16).numpy())
        if ks is not None:
            assert np.array_equal(many[2].view(np.uint32), ks.numpy().view(np.uint32))
            assert np.array_equal(many[3].view(np.uint32), vs.numpy().view(np.uint32))


def test_append_of_several_tokens_equals_single_token_appends():
    check_multi_token_append()


PINS = (check_encoder, check_round_trip, check_saturation_and_zeros, check_bf16_append, check_fp8_append,
        check_error_masks, check_multi_token_append)


def test_encoder_matches_torch_on_every_rounding_boundary():
    check_encoder()


def test_encoder_round_trips_every_finite_code():
    check_round_trip()


def test_encoder_saturates_and_keeps_signed_zeros():
    check_saturation_and_zeros()


def test_bf16_append_writes_exactly_the_target_slots():
    check_bf16_append()


def test_fp8_append_matches_the_generator_quantiser_and_error_bound():
    check_fp8_append()


def test_append_reports_bad_positions_and_pages():
    check_error_masks()


def test_row_kinds_cover_the_special_rows():
    rows = inputs.new_token_rows(16, seed=3).to(torch.float32).numpy()
    assert np.all(rows[1] == 0) and np.all(rows[2] == 0) and np.signbit(rows[2]).any()
    assert np.abs(rows[5]).max() > 1e29 and np.abs(rows[6]).max() < 1e-28
    assert (np.abs(rows[3]) < 2.0 ** -6 * np.abs(rows[3]).max() / 448).any()


_MUTANTS = {
    "ties_down": ("(dist == bd && (c & 1) == 0)", "(dist == bd && 0)"),
    "ties_up": ("(dist == bd && (c & 1) == 0)", "(dist == bd)"),
    "overflow_nan": ("int best = 0x7E;", "int best = 0x7F;"),
    "sign_dropped": ("neg ? (0x80 | best) : best", "best"),
    "scale_447": ("absmax / 448.0f", "absmax / 447.0f"),
    "mul_not_div": ("bf16_to_float(x[i]) / s)", "bf16_to_float(x[i]) * s)"),
    "zero_row_scale": (": 1.0f;", ": 0.5f;"),
    "absmax_first": ("if (a > absmax) absmax = a;", "if (i == 0) absmax = a;"),
    "wrong_slot": ("(size_t)(t % page)", "(size_t)((t + 1) % page)"),
    "wrong_page": ("t / page]", "(t / page + 1) % max_pages]"),
    "k_for_v": ("quantise_row(v_new + (size_t)x * d", "quantise_row(k_new + (size_t)x * d"),
    "token_offset_dropped": ("positions[b] + x % T;", "positions[b];"),
    "bf16_v_from_k": ("memcpy((uint16_t *)v_cache + row * d, v_new", "memcpy((uint16_t *)v_cache + row * d, k_new"),
    "position_not_reported": ("mask |= 2;", "mask |= 0;"),
    "block_not_reported": ("mask |= 1;", "mask |= 0;"),
}


def _pins_pass(lib) -> bool:
    try:
        for pin in PINS:
            pin(lib)
    except AssertionError:
        return False
    return True


def test_append_mutants_are_caught():
    src = open(os.path.join(os.path.dirname(oracle.__file__), "mfa_oracle.c")).read()
    assert _pins_pass(oracle._load())
    with tempfile.TemporaryDirectory() as tmp:
        for name, (old, new) in _MUTANTS.items():
            assert src.count(old) >= 1, f"mutant {name}: pattern not found"
            path = os.path.join(tmp, f"{name}.c")
            with open(path, "w") as f:
                f.write(src.replace(old, new))
            so = os.path.join(tmp, f"{name}.so")
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                                   "-fno-fast-math", "-ffp-contract=off", "-o", so, path, "-lm"])
            assert not _pins_pass(oracle.load_library(so)), f"mutant {name} survived the pins"


