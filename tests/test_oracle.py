"""Pins for the CPU oracle: each check ties it to something other than itself.

The decode step is softmax(q K^T * scale) V over a paged cache with one shared
K head and one shared V head (Step-3, paperlayer.ai/abs/2507.19427v1, section 2
"Step-3 Model Card" and section 5 "Model-System Co-design").  The pages print no
worked example, so the pins are library routines (torch SDPA, scipy
logsumexp, torch's float8_e4m3fn decoder), closed forms and invariants that
the definition fixes.  ``test_mutants_are_caught`` plants mistakes in copies
of the oracle and checks that these pins reject every one.
"""
import math
import os
import subprocess
import tempfile

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from decode_attention_02_gb300 import inputs

TOL = 1e-12


def dense_kv(case, b):
    """Gather sequence b's keys and values by numpy indexing, decoded by torch: [L, G*d] rows
    (G key/value heads side by side; the values are the keys when the latent is shared)."""
    w = case.workload
    L = int(case.seq_lens[b])
    t = np.arange(L)
    blk = case.block_table.numpy()[b, t // w.page_size]
    slot = t % w.page_size
    if w.kv_dtype == "bf16":
        K = case.k_cache[blk, slot].to(torch.float64)
        V = case.v_cache[blk, slot].to(torch.float64)
    elif w.kv_dtype == "mxfp4":
        K = mx_dense(case.k_cache[blk, slot], case.k_scale[blk, slot])
        V = mx_dense(case.v_cache[blk, slot], case.v_scale[blk, slot])
    else:
        K = case.k_cache[blk, slot].view(torch.float8_e4m3fn).to(torch.float64) * \
            case.k_scale[blk, slot].to(torch.float64)[:, None]
        V = case.v_cache[blk, slot].view(torch.float8_e4m3fn).to(torch.float64) * \
            case.v_scale[blk, slot].to(torch.float64)[:, None]
    if getattr(w, "kv_shared", False):
        V = K.clone()
    return K, V


# OCP MX FP4 (E2M1) magnitudes by code 0..7; codes 8..15 are their negatives
E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def mx_dense(codes, scales):
    """MXFP4 rows (uint8 [..., n/2] nibble pairs, element 2i in the low nibble; E8M0 uint8
    [..., n/32]) -> float64 [..., n]: the E2M1 value times its block's scale, the scale
    decoded by torch's float8_e8m0fnu."""
    c = codes.numpy()
    full = np.empty(c.shape[:-1] + (2 * c.shape[-1],), dtype=np.uint8)
    full[..., 0::2], full[..., 1::2] = c & 15, c >> 4
    s = scales.contiguous().view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    return torch.from_numpy(E2M1_VALUES[full] * np.repeat(s, 32, axis=-1))


def sdpa_reference(case, scale=None):
    """torch SDPA (float64) on the dense gather, and scipy logsumexp of the scores.  With G
    key/value heads, the [L, G*d] rows are split into heads and each repeated for its H/G
    query heads (query head h reads head h // (H/G))."""
    w = case.workload
    scale = w.scale() if scale is None else scale
    B, H, d = case.q.shape
    G = getattr(w, "num_kv_heads", 1)
    out = np.zeros((B, H, d))
    lse = np.full((B, H), -np.inf)
    for b in range(B):
        K, V = dense_kv(case, b)
        if K.shape[0] == 0:
            continue
        Kh = K.view(-1, G, d).permute(1, 0, 2).repeat_interleave(H // G, dim=0)   # [H, L, d]
        Vh = V.view(-1, G, d).permute(1, 0, 2).repeat_interleave(H // G, dim=0)
        q = case.q[b].to(torch.float64)
        o = torch.nn.functional.scaled_dot_product_attention(
            q[None, :, None, :], Kh[None], Vh[None], scale=scale)
        out[b] = o[0, :, 0, :].numpy()
        scores = np.einsum("hd,hld->hl", q.numpy(), Kh.numpy()) * scale
        lse[b] = scipy.special.logsumexp(scores, axis=1)
    return out, lse


def assert_close(a, b, tol=TOL):
    a, b = np.asarray(a), np.asarray(b)
    assert a.shape == b.shape
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        diff = np.where(both_inf, 0.0, np.abs(a - b))
    assert np.all(np.isfinite(diff)), "non-finite mismatch"
    assert diff.max(initial=0.0) <= tol, f"max diff {diff.max()} > {tol}"


# ---------------------------------------------------------------- format pins

def test_e4m3_every_code_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])
    # spot values of the format: max normal, min normal, min subnormal, signed zero
    assert oracle.e4m3_to_double(0x7E) == 448.0
    assert oracle.e4m3_to_double(0x08) == 2.0 ** -6
    assert oracle.e4m3_to_double(0x01) == 2.0 ** -9
    assert oracle.e4m3_to_double(0xFE) == -448.0


# ------------------------------------------------------- library-routine pins

@pytest.mark.parametrize("lens", [[1, 65, 200], [63, 64, 130, 0], [129, 7]])
def test_matches_sdpa_full_shape(lens):
    case = inputs.small("sdpa", len(lens), lens, seed=11 + len(lens))
    out, lse = oracle.decode(case)
    ref_o, ref_lse = sdpa_reference(case)
    assert_close(out, ref_o)
    assert_close(lse, ref_lse)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_sdpa_tiny_shapes(seed):
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, 131, size=3).tolist()
    case = inputs.small("tiny", 3, lens, seed=seed, num_q_heads=4, head_dim=8, page_size=4)
    out, lse = oracle.decode(case)
    ref_o, ref_lse = sdpa_reference(case)
    assert_close(out, ref_o)
    assert_close(lse, ref_lse)


def test_matches_sdpa_fp8():
    case = inputs.small("fp8", 3, [1, 100, 257], kv_dtype="fp8_e4m3", seed=21)
    out, lse = oracle.decode(case)
    ref_o, ref_lse = sdpa_reference(case)
    assert_close(out, ref_o)
    assert_close(lse, ref_lse)


def test_softmax_scale_is_honoured():
    case = inputs.small("scale", 2, [77, 150], seed=31)
    out, lse = oracle.decode(case, softmax_scale=0.3)
    ref_o, ref_lse = sdpa_reference(case, scale=0.3)
    assert_close(out, ref_o)
    assert_close(lse, ref_lse)


def test_spiked_keys_match_sdpa():
    case = inputs.small("spike", 2, [300, 64], seed=41, k_spike_frac=0.01)
    out, lse = oracle.decode(case)
    ref_o, ref_lse = sdpa_reference(case)
    assert_close(out, ref_o, 1e-11)
    assert_close(lse, ref_lse, 1e-11)


# ---------------------------------------------------------- closed-form pins

def test_length_one_returns_v0_exactly():
    case = inputs.small("l1", 2, [1, 1], seed=51)
    out, lse = oracle.decode(case)
    for b in range(2):
        K, V = dense_kv(case, b)
        assert np.array_equal(out[b], np.broadcast_to(V[0].numpy(), out[b].shape))
        s0 = (case.q[b].to(torch.float64).numpy() @ K[0].numpy()) * case.workload.scale()
        assert_close(lse[b], s0)


def test_two_tokens_logistic_closed_form():
    case = inputs.small("l2", 3, [2, 2, 2], seed=61)
    out, lse = oracle.decode(case)
    for b in range(3):
        K, V = dense_kv(case, b)
        q = case.q[b].to(torch.float64).numpy()
        s = (q @ K.numpy().T) * case.workload.scale()          # [H, 2]
        w0 = scipy.special.expit(s[:, 0] - s[:, 1])
        w1 = scipy.special.expit(s[:, 1] - s[:, 0])
        ref = w0[:, None] * V[0].numpy()[None] + w1[:, None] * V[1].numpy()[None]
        assert_close(out[b], ref, 1e-14)
        assert_close(lse[b], np.logaddexp(s[:, 0], s[:, 1]))


def _fill_used_rows(case, b, rows, which):
    """Write ``rows`` [L, d] (bf16) into sequence b's slots of the K or V pool."""
    w = case.workload
    pool = case.k_cache if which == "k" else case.v_cache
    L = int(case.seq_lens[b])
    for t in range(L):
        blk = int(case.block_table[b, t // w.page_size])
        pool[blk, t % w.page_size] = rows[t]


def test_constant_keys_give_mean_of_values():
    case = inputs.small("constk", 2, [97, 200], seed=71)
    for b in range(2):
        L = int(case.seq_lens[b])
        row = case.k_cache[int(case.block_table[b, 0]), 0].clone()
        _fill_used_rows(case, b, row.expand(L, -1), "k")
    out, lse = oracle.decode(case)
    for b in range(2):
        K, V = dense_kv(case, b)
        assert_close(out[b], np.broadcast_to(V.numpy().mean(axis=0), out[b].shape), 1e-13)
        s = (case.q[b].to(torch.float64).numpy() @ K[0].numpy()) * case.workload.scale()
        assert_close(lse[b], s + math.log(K.shape[0]), 1e-12)


def test_constant_values_are_returned():
    case = inputs.small("constv", 2, [50, 130], seed=81)
    u = torch.randn(case.workload.head_dim, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    for b in range(2):
        _fill_used_rows(case, b, u.expand(int(case.seq_lens[b]), -1), "v")
    out, _ = oracle.decode(case)
    assert_close(out, np.broadcast_to(u.to(torch.float64).numpy(), out.shape), 1e-14)


def test_output_lies_in_convex_hull_of_values():
    case = inputs.small("hull", 3, [5, 64, 333], seed=91)
    out, _ = oracle.decode(case)
    for b in range(3):
        _, V = dense_kv(case, b)
        lo, hi = V.numpy().min(axis=0), V.numpy().max(axis=0)
        assert np.all(out[b] >= lo - 1e-12) and np.all(out[b] <= hi + 1e-12)


# ------------------------------------------------------------ invariance pins

def test_block_permutation_is_bitwise_invariant():
    case = inputs.small("perm", 3, [10, 64, 250], seed=101, extra_blocks=3)
    out, lse = oracle.decode(case)
    nb = case.num_blocks
    perm = torch.from_numpy(np.random.default_rng(5).permutation(nb))
    k2 = torch.empty_like(case.k_cache)
    v2 = torch.empty_like(case.v_cache)
    k2[perm] = case.k_cache
    v2[perm] = case.v_cache
    table = case.block_table.clone()
    used = table >= 0
    table[used] = perm[table[used].long()].to(torch.int32)
    case2 = inputs.Case(case.workload, case.q, k2, v2, None, None, table, case.seq_lens)
    out2, lse2 = oracle.decode(case2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_token_permutation_invariance():
    case = inputs.small("tperm", 2, [129, 200], seed=111)
    out, lse = oracle.decode(case)
    for b in range(2):
        K, V = dense_kv(case, b)
        p = torch.from_numpy(np.random.default_rng(b).permutation(K.shape[0]))
        _fill_used_rows(case, b, K[p].to(torch.bfloat16), "k")
        _fill_used_rows(case, b, V[p].to(torch.bfloat16), "v")
    out2, lse2 = oracle.decode(case)
    assert_close(out, out2, 1e-13)
    assert_close(lse, lse2, 1e-12)


def test_key_shift_invariance():
    # keys on an exact grid (j/8, |j| <= 64) so that k_t + c stays exact in bf16
    case = inputs.small("shift", 2, [40, 150], seed=121)
    g = np.random.default_rng(7)
    d = case.workload.head_dim
    c = torch.from_numpy(g.integers(-64, 65, size=d) / 8.0).to(torch.bfloat16)
    for b in range(2):
        L = int(case.seq_lens[b])
        base = torch.from_numpy(g.integers(-64, 65, size=(L, d)) / 8.0).to(torch.bfloat16)
        _fill_used_rows(case, b, base, "k")
    out, lse = oracle.decode(case)
    for b in range(2):
        K, _ = dense_kv(case, b)
        shifted = (K + c.to(torch.float64)[None]).to(torch.bfloat16)
        assert torch.equal(shifted.to(torch.float64), K + c.to(torch.float64)[None])
        _fill_used_rows(case, b, shifted, "k")
    out2, lse2 = oracle.decode(case)
    assert_close(out, out2, 1e-12)
    shift = (case.q.to(torch.float64).numpy() @ c.to(torch.float64).numpy()) * case.workload.scale()
    assert_close(lse2 - lse, shift, 1e-10)


# ------------------------------------------------------------- split / merge

@pytest.mark.parametrize("seed", [0, 1])
def test_split_then_merge_equals_one_pass(seed):
    case = inputs.small("split", 3, [1, 200, 517], seed=131 + seed)
    out, lse = oracle.decode(case)
    rng = np.random.default_rng(seed)
    S = 4
    cuts = []
    for b in range(3):
        L = int(case.seq_lens[b])
        c = np.sort(rng.integers(0, L + 1, size=S - 1))
        cuts.append(np.concatenate([[0], c, [L]]))
    cuts = np.array(cuts)
    po, pl = [], []
    for s in range(S):
        o, l_ = oracle.decode(case, t_begin=cuts[:, s], t_end=cuts[:, s + 1])
        po.append(o)
        pl.append(l_)
    mo, ml = oracle.combine(np.stack(po), np.stack(pl))
    assert_close(mo, out, 1e-12)
    assert_close(ml, lse, 1e-12)


def test_combine_of_all_empty_partials():
    po = np.zeros((3, 2, 4, 8))
    pl = np.full((3, 2, 4), -np.inf)
    o, l_ = oracle.combine(po, pl)
    assert np.all(o == 0) and np.all(np.isneginf(l_))


# ---------------------------------------------------------------- edge cases

def test_empty_sequence_gives_zero_and_minus_inf():
    case = inputs.small("empty", 3, [0, 5, 0], seed=141)
    out, lse = oracle.decode(case)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    assert np.all(np.isneginf(lse[0])) and np.all(np.isneginf(lse[2]))
    assert np.all(np.isfinite(out[1])) and np.all(np.isfinite(lse[1]))


def test_poisoned_slots_are_never_read():
    for kv in ("bf16", "fp8_e4m3"):
        case = inputs.small("poison", 3, [3, 64, 190], kv_dtype=kv, seed=151, extra_blocks=4)
        out, lse = oracle.decode(case)
        assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))


def test_thread_count_does_not_change_results():
    case = inputs.small("threads", 3, [100, 3, 260], seed=161)
    a = oracle.decode(case, nthreads=1)
    b = oracle.decode(case, nthreads=5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ------------------------------------------------------------- mutation check

_MUTANTS = {
    "wrong_slot": ("(size_t)(t % J->page)", "(size_t)((t + 1) % J->page)"),
    "wrong_block": ("t / J->page]", "(t / J->page + 1) % J->max_pages]"),
    "k_for_v": ("kv_row(J, 1, b, t, g, W->row);", "kv_row(J, 0, b, t, g, W->row);"),
    "sign_flip": ("(t - t0)] - m[h - h0])", "(t - t0)] * -1.0 + m[h - h0])"),
    "no_scale": ("double st = J->scale * acc;", "double st = acc;"),
    "lse_no_log": ("m[h - h0] + log(l[h - h0])", "m[h - h0] + l[h - h0]"),
    "no_normalise": ("o[i] /= l[h - h0];", "o[i] /= 1.0;"),
    "e4m3_bias": ("e - 7)", "e - 8)"),
    "e4m3_subnormal": ("(double)m / 8.0, -6)", "(double)m / 8.0, -7)"),
    "fp8_scale_dropped": ("* (double)sc[row]", "* 1.0"),
    "head_index": ("W->q[(size_t)(h - h0) * d + i] = bf16_to_double(qh[i]);",
                   "W->q[(size_t)(h - h0) * d + i] = bf16_to_double(qh[i % 8]);"),
    # grouped and shared key/value heads
    "group_interleaved": ("int g = h0 / (J->H / J->G);", "int g = (h0 / HEAD_GROUP) % J->G;"),
    "row_width_dropped": ("row * (size_t)J->G * (size_t)J->d", "row * (size_t)J->d"),
    "values_always_keys": ("const void *vpool = J->v_cache ? J->v_cache : J->k_cache;",
                           "const void *vpool = J->k_cache;"),
}


def _run_pins(lib):
    """The library/closed-form pins, on a fresh library; returns True if all pass."""
    try:
        codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
        ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
        got = np.array([oracle.e4m3_to_double(c, lib=lib) for c in range(256)])
        m = ~np.isnan(ref)
        if not np.array_equal(ref[m], got[m]):
            return False
        for kv in ("bf16", "fp8_e4m3"):
            case = inputs.small("mut", 2, [70, 131], kv_dtype=kv, seed=171)
            out, lse = oracle.decode(case, lib=lib)
            ro, rl = sdpa_reference(case)
            assert_close(out, ro)
            assert_close(lse, rl)
        for kw in (dict(num_q_heads=32, head_dim=16, num_kv_heads=2), dict(num_q_heads=8, head_dim=32, kv_shared=True)):
            case = inputs.small("mutg", 2, [70, 131], seed=172, **kw)
            out, lse = oracle.decode(case, lib=lib)
            ro, rl = sdpa_reference(case)
            assert_close(out, ro)
            assert_close(lse, rl)
    except AssertionError:
        return False
    return True


def test_mutants_are_caught():
    src = open(os.path.join(os.path.dirname(oracle.__file__), "mfa_oracle.c")).read()
    assert _run_pins(oracle._load())
    with tempfile.TemporaryDirectory() as tmp:
        for name, (old, new) in _MUTANTS.items():
            assert src.count(old) >= 1, f"mutant {name}: pattern not found"
            path = os.path.join(tmp, f"{name}.c")
            with open(path, "w") as f:
                f.write(src.replace(old, new))
            so = os.path.join(tmp, f"{name}.so")
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                                   "-o", so, path, "-lm"])
            assert not _run_pins(oracle.load_library(so)), f"mutant {name} survived the pins"


# ------------------------------------------------------------- multi-token decode

def dense_mtp_reference(case):
    """Multi-token decode written with an explicit causal mask over a dense gather: the T new
    tokens are the last T cached ones, and query token i may see key t only if t <= L - T + i."""
    w = case.workload
    T = w.tokens_per_seq
    B = case.seq_lens.shape[0]
    H, d = case.q.shape[1], case.q.shape[2]
    out = np.zeros((B * T, H, d))
    lse = np.full((B * T, H), -np.inf)
    for b in range(B):
        L = int(case.seq_lens[b])
        if L == 0:
            continue
        K, V = dense_kv(case, b)
        K, V = K.numpy(), V.numpy()
        for i in range(T):
            q = case.q[b * T + i].to(torch.float64).numpy()
            s = (q @ K.T) * w.scale()                      # [H, L]
            visible = np.arange(L) <= L - T + i
            if not visible.any():
                continue
            s = np.where(visible[None, :], s, -np.inf)
            lse[b * T + i] = scipy.special.logsumexp(s, axis=1)
            out[b * T + i] = np.exp(s - lse[b * T + i][:, None]) @ V
    return out, lse


@pytest.mark.parametrize("T", [2, 3, 4])
@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_multi_token_decode_matches_an_explicit_causal_mask(T, kv):
    case = inputs.small("mtp", 5, [1, 2, 65, 130, 3], kv_dtype=kv, seed=170 + T, tokens_per_seq=T)
    out, lse = oracle.decode(case)
    ro, rl = dense_mtp_reference(case)
    assert_close(out, ro)
    assert np.array_equal(np.isneginf(lse), np.isneginf(rl))
    fin = np.isfinite(rl)
    assert np.abs(lse[fin] - rl[fin]).max() <= TOL


def test_multi_token_decode_last_token_is_the_ordinary_decode():
    """Query token T - 1 sees the whole cache: it is the single-token decode of its q."""
    T = 3
    case = inputs.small("mtp_last", 4, [7, 64, 200, 129], seed=183, tokens_per_seq=T)
    out, lse = oracle.decode(case)
    single = inputs.Case(workload=inputs.Workload("single", batch=4, lens=(7, 64, 200, 129)),
                         q=case.q[T - 1::T].contiguous(), k_cache=case.k_cache, v_cache=case.v_cache,
                         k_scale=None, v_scale=None, block_table=case.block_table, seq_lens=case.seq_lens)
    o1, l1 = oracle.decode(single)
    assert np.array_equal(out[T - 1::T], o1) and np.array_equal(lse[T - 1::T], l1)


# ------------------------------------------------------------- ablation shapes

@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_grouped_query_heads_match_sdpa_with_explicit_grouping(kv):
    """GQA-style cache at the ablation shape: 64 query heads over 4 key/value heads of width
    128 (rows of 4 x 128), against torch SDPA with each head's keys and values repeated for
    its 16 query heads."""
    case = inputs.small("gqa", 3, [1, 70, 200], kv_dtype=kv, seed=190, head_dim=128, num_kv_heads=4)
    assert case.k_cache.shape[2] == 4 * 128
    out, lse = oracle.decode(case)
    ro, rl = sdpa_reference(case)
    assert_close(out, ro)
    assert_close(lse, rl)


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_shared_latent_matches_sdpa_with_values_equal_to_keys(kv):
    """MLA-style cache at the ablation shape: 128 query heads over one 512-wide latent that
    serves as keys and values (no V pool), against torch SDPA with V = K."""
    case = inputs.small("mla", 2, [5, 131], kv_dtype=kv, seed=191, num_q_heads=128, head_dim=512,
                        kv_shared=True)
    assert case.v_cache is case.k_cache
    out, lse = oracle.decode(case)
    ro, rl = sdpa_reference(case)
    assert_close(out, ro)
    assert_close(lse, rl)


def test_grouped_heads_see_only_their_own_key_value_head():
    """Changing key/value head 2's columns of every cache row changes exactly query heads
    32..47 (the 16 heads that read head 2)."""
    case = inputs.small("gqa_iso", 2, [90, 33], seed=192, head_dim=128, num_kv_heads=4)
    out, lse = oracle.decode(case)
    k2 = case.k_cache.clone()
    v2 = case.v_cache.clone()
    k2[:, :, 256:384] = k2[:, :, 256:384].flip(1)
    v2[:, :, 256:384] = -v2[:, :, 256:384]
    mod = inputs.Case(workload=case.workload, q=case.q, k_cache=k2, v_cache=v2, k_scale=None, v_scale=None,
                      block_table=case.block_table, seq_lens=case.seq_lens)
    out2, lse2 = oracle.decode(mod)
    same = np.array([np.array_equal(out[:, h], out2[:, h]) for h in range(64)])
    assert same[:32].all() and same[48:].all() and not same[32:48].any()


def test_shared_latent_equals_separate_pools_holding_the_same_rows():
    """A shared latent gives bitwise the same result as a V pool that is a copy of the K pool."""
    case = inputs.small("mla_eq", 2, [64, 200], seed=193, num_q_heads=16, head_dim=64, kv_shared=True)
    import dataclasses
    sep = inputs.Case(workload=dataclasses.replace(case.workload, kv_shared=False), q=case.q,
                      k_cache=case.k_cache, v_cache=case.k_cache.clone(), k_scale=None, v_scale=None,
                      block_table=case.block_table, seq_lens=case.seq_lens)
    a, b = oracle.decode(case), oracle.decode(sep)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
