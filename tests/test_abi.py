"""Host-side checks of the C ABI (no GPU needed): exports, validation, planning."""
import ctypes
import re
import os

import pytest

import decode_attention_02_gb300 as mfa
from decode_attention_02_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return mfa.load_library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "mfa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mfa_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(names) == set(mfa.EXPORTED_SYMBOLS)
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
    assert lib.mfa_abi_version() == 5


def test_status_strings(lib):
    for s in range(6):
        assert mfa.status_string(s) not in ("", "unknown status")
    assert mfa.status_string(99) == "unknown status"


def problem(**kw):
    args = dict(batch=4, max_pages_per_seq=8, num_blocks=32)
    args.update(kw)
    return mfa.make_problem(**args)


def test_plan_one_cta_per_sm_when_enough_tiles(lib):
    p = problem(batch=32, max_pages_per_seq=64, num_blocks=2048)
    plan = mfa.mfa_decode_plan(p, [4096] * 32, num_sms=152)
    assert plan.num_ctas == 152
    assert plan.total_tiles == 32 * 32
    assert plan.max_tiles_per_cta == 7          # 1024 tiles and 31 boundaries over 152 CTAs
    assert plan.num_partials == 32 + 152 - 1
    o_off, l_off = mfa.workspace_layout(plan)
    assert plan.workspace_bytes >= l_off + plan.num_partials * 64 * 4
    assert o_off == 256 and l_off % 256 == 0 and plan.workspace_bytes % 256 == 0


def split_tiles_brute_force(lens, G, c):
    """Tiles per CTA under the documented split, by enumerating every tile: tile k of sequence
    b at cost 4 (S_b + k) + c N_b, owned by the largest g with floor(g C / G) <= its cost."""
    tiles = [(L + 127) // 128 for L in lens]
    W, N = sum(tiles), sum(1 for t in tiles if t > 0)
    C = 4 * W + c * max(N - 1, 0)
    per = [0] * G
    before = nonempty = 0
    for t in tiles:
        for k in range(t):
            x = 4 * (before + k) + c * nonempty
            per[max(g for g in range(G) if (g * C) // G <= x)] += 1
        before += t
        nonempty += t > 0
    return per


@pytest.mark.parametrize("kv, c", [(mfa.MFA_KV_BF16, 3), (mfa.MFA_KV_FP8_E4M3, 10), (mfa.MFA_KV_MXFP4, 10)])
def test_plan_tile_counts_follow_the_documented_split(lib, kv, c):
    import random
    rng = random.Random(5)
    for trial in range(40):
        B = rng.randint(1, 40)
        lens = [rng.choice([0, 1, 64, 128, 129, rng.randint(0, 4096)]) for _ in range(B)]
        G = rng.randint(1, 60)
        plan = mfa.mfa_decode_plan(problem(batch=B, max_pages_per_seq=64, num_blocks=4096, kv_dtype=kv), lens,
                                   num_sms=152, force_ctas=G)
        per = split_tiles_brute_force(lens, G, c)
        assert sum(per) == plan.total_tiles
        assert plan.max_tiles_per_cta == max(per), (lens, G)
    # the boundary weight moves tiles away from CTAs that hold a sequence switch
    lens = [4096] * 32
    plan = mfa.mfa_decode_plan(problem(batch=32, max_pages_per_seq=64, num_blocks=2048, kv_dtype=kv), lens,
                               num_sms=152)
    assert plan.max_tiles_per_cta == max(split_tiles_brute_force(lens, 152, c))


@pytest.mark.parametrize("kv, c", [(mfa.MFA_KV_BF16, 3), (mfa.MFA_KV_FP8_E4M3, 10)])
def test_multi_token_plan_walks_the_units_reader_major(lib, kv, c):
    """T query tokens a sequence: the units are laid end to end reader-major (every sequence's
    token 0, then every sequence's token 1, ...), token i of a sequence of L seeing L - T + 1 + i
    tokens.  The plan's largest CTA share is the documented split over that order, and for
    some of these ragged mixes it differs from the split over the sequence-major order."""
    import random
    rng = random.Random(11)
    differs = 0
    for trial in range(30):
        B, T = rng.randint(1, 24), rng.randint(2, 4)
        lens = [rng.choice([0, 1, 2, 130, rng.randint(0, 3000)]) for _ in range(B)]
        vis = lambda b, i: max(0, lens[b] - (T - 1 - i))
        reader_major = [vis(b, i) for i in range(T) for b in range(B)]
        seq_major = [vis(b, i) for b in range(B) for i in range(T)]
        W = sum((L + 127) // 128 for L in reader_major)
        G = rng.randint(max(1, -(-W // 96)), max(2, -(-W // 96)) + 40)   # room under the 128-tile cap
        plan = mfa.mfa_decode_plan(problem(batch=B, max_pages_per_seq=64, num_blocks=4096, kv_dtype=kv,
                                           tokens_per_seq=T), lens, num_sms=152, force_ctas=G)
        per = split_tiles_brute_force(reader_major, G, c)
        assert sum(per) == plan.total_tiles
        assert plan.max_tiles_per_cta == max(per), (lens, T, G)
        differs += max(split_tiles_brute_force(seq_major, G, c)) != max(per)
    assert differs > 0


def test_plan_fewer_ctas_than_sms_for_short_batches(lib):
    plan = mfa.mfa_decode_plan(problem(batch=1), [512], num_sms=152)
    assert plan.num_ctas == 4 and plan.max_tiles_per_cta == 1
    plan = mfa.mfa_decode_plan(problem(batch=2), [0, 0], num_sms=152)
    assert plan.num_ctas == 1


def test_plan_without_host_lengths_uses_the_bound(lib):
    plan = mfa.mfa_decode_plan(problem(batch=4, max_pages_per_seq=8), None, max_seq_len=300, num_sms=152)
    assert plan.total_tiles == 4 * 3


def test_plan_caps_tiles_per_cta(lib):
    p = problem(batch=4, max_pages_per_seq=2048, num_blocks=8192)
    plan = mfa.mfa_decode_plan(p, [131072] * 4, num_sms=2)
    # 4096 tiles: 32 CTAs would be the floor, but the sequence boundaries' cost leaves one of
    # them 129 tiles, so the plan takes the smallest count that fits
    assert plan.max_tiles_per_cta <= 128 and plan.num_ctas == 33
    with pytest.raises(mfa.MfaError):
        mfa.mfa_decode_plan(p, [131072] * 4, num_sms=2, force_ctas=2)


def test_plan_from_a_bound_fits_any_shorter_lengths(lib):
    # planned for B sequences of at most max_seq_len tokens, the grid must keep every CTA
    # within 128 tiles whatever the actual mix: its cost range of ceil(C / G) units holds
    # at most ceil(ceil(C / G) / 4) tiles, C = 4 W + 3 (B - 1)
    p = problem(batch=4, max_pages_per_seq=2048, num_blocks=8192)
    plan = mfa.mfa_decode_plan(p, None, max_seq_len=131072, num_sms=2)
    C = 4 * 4096 + 3 * 3
    G = plan.num_ctas
    assert (-(-C // G) + 3) // 4 <= 128 and (-(-C // (G - 1)) + 3) // 4 > 128


def test_plan_rejects_bad_input(lib):
    with pytest.raises(mfa.MfaError) as e:
        mfa.mfa_decode_plan(problem(), [1, 2, 3, 10 ** 6], num_sms=8)
    assert e.value.status == mfa.MFA_ERR_INVALID_ARG
    for bad, code in [(dict(num_q_heads=32), mfa.MFA_ERR_UNSUPPORTED),
                      (dict(head_dim=128), mfa.MFA_ERR_UNSUPPORTED),
                      (dict(page_size=16), mfa.MFA_ERR_UNSUPPORTED),
                      (dict(softmax_scale=0.0), mfa.MFA_ERR_INVALID_ARG),
                      (dict(softmax_scale=float("nan")), mfa.MFA_ERR_INVALID_ARG),
                      (dict(kv_dtype=7), mfa.MFA_ERR_INVALID_ARG),
                      (dict(out_dtype=2), mfa.MFA_ERR_INVALID_ARG),
                      (dict(batch=-1), mfa.MFA_ERR_INVALID_ARG),
                      (dict(num_blocks=0), mfa.MFA_ERR_INVALID_ARG),
                      # shapes: only MFA, the grouped-head shape and the shared latent are built,
                      # the last two for a bf16 cache and one query token
                      (dict(num_kv_heads=2), mfa.MFA_ERR_UNSUPPORTED),
                      (dict(num_kv_heads=0), mfa.MFA_ERR_INVALID_ARG),
                      (dict(kv_shared=True), mfa.MFA_ERR_UNSUPPORTED),
                      (dict(head_dim=128, num_kv_heads=4, kv_dtype=mfa.MFA_KV_FP8_E4M3), mfa.MFA_ERR_UNSUPPORTED),
                      (dict(head_dim=128, num_kv_heads=4, tokens_per_seq=2), mfa.MFA_ERR_UNSUPPORTED),
                      (dict(num_q_heads=128, head_dim=512), mfa.MFA_ERR_UNSUPPORTED),
                      (dict(num_q_heads=128, head_dim=512, kv_shared=True, kv_dtype=mfa.MFA_KV_FP8_E4M3),
                       mfa.MFA_ERR_UNSUPPORTED),
                      (dict(head_dim=128, num_kv_heads=4, kv_dtype=mfa.MFA_KV_MXFP4), mfa.MFA_ERR_UNSUPPORTED),
                      (dict(kv_dtype=3), mfa.MFA_ERR_INVALID_ARG)]:
        with pytest.raises(mfa.MfaError) as e:
            mfa.mfa_decode_plan(problem(**bad), None, max_seq_len=64, num_sms=8)
        assert e.value.status == code, bad


def test_plan_for_the_comparison_shapes(lib):
    """Grouped heads: one 64-head unit per sequence, 128-wide partials; shared latent: two
    64-head units per sequence (128 query heads), 512-wide partials."""
    lens = [4096, 100, 0]
    g = mfa.mfa_decode_plan(problem(batch=3, head_dim=128, num_kv_heads=4, max_pages_per_seq=64), lens, num_sms=8)
    assert g.total_tiles == 32 + 1 and g.num_partials == 3 + g.num_ctas - 1
    o, l = mfa.workspace_layout(g, head_dim=128)
    assert l == (256 + g.num_partials * 64 * 128 * 4 + 255) // 256 * 256
    assert g.workspace_bytes == (l + g.num_partials * 64 * 4 + 255) // 256 * 256
    m = mfa.mfa_decode_plan(problem(batch=3, num_q_heads=128, head_dim=512, kv_shared=True, max_pages_per_seq=64),
                            lens, num_sms=8)
    assert m.total_tiles == 2 * (32 + 1) and m.num_partials == 6 + m.num_ctas - 1
    o, l = mfa.workspace_layout(m, head_dim=512)
    assert m.workspace_bytes == (l + m.num_partials * 64 * 4 + 255) // 256 * 256


def _run_raw(lib, plan, prob, ptrs, ws_bytes):
    P = ctypes.c_void_p
    return lib.mfa_decode_run(ctypes.byref(plan), ctypes.byref(prob), *[P(x) if x else None for x in ptrs],
                              ctypes.c_uint64(ws_bytes), None)


def test_run_validates_before_touching_the_device(lib):
    prob = problem()
    plan = mfa.mfa_decode_plan(prob, [10, 20, 30, 40], num_sms=8)
    good = [0x1000, 0x2000, 0x3000, None, None, 0x4000, 0x5000, 0x6000, 0x7000, 0x10000]
    # q, k, v, k_scale, v_scale, table, lens, out, lse, workspace
    bad_null = list(good); bad_null[0] = None
    assert _run_raw(lib, plan, prob, bad_null, plan.workspace_bytes) == mfa.MFA_ERR_INVALID_ARG
    bad_align = list(good); bad_align[1] = 0x2008
    assert _run_raw(lib, plan, prob, bad_align, plan.workspace_bytes) == mfa.MFA_ERR_INVALID_ARG
    bad_ws = list(good); bad_ws[9] = 0x10010
    assert _run_raw(lib, plan, prob, bad_ws, plan.workspace_bytes) == mfa.MFA_ERR_INVALID_ARG
    assert _run_raw(lib, plan, prob, good, plan.workspace_bytes - 1) == mfa.MFA_ERR_WORKSPACE
    other = problem(batch=5)
    assert _run_raw(lib, plan, other, good, plan.workspace_bytes) == mfa.MFA_ERR_INVALID_ARG
    # an MXFP4 cache needs both scale arrays, 16-byte aligned (their pages are bulk copies)
    mxp = problem(kv_dtype=mfa.MFA_KV_MXFP4)
    mplan = mfa.mfa_decode_plan(mxp, [10, 20, 30, 40], num_sms=8)
    assert _run_raw(lib, mplan, mxp, good, mplan.workspace_bytes) == mfa.MFA_ERR_INVALID_ARG
    mgood = list(good); mgood[3], mgood[4] = 0x8000, 0x9000
    mbad = list(mgood); mbad[4] = 0x9008
    assert _run_raw(lib, mplan, mxp, mbad, mplan.workspace_bytes) == mfa.MFA_ERR_INVALID_ARG


def _append_raw(lib, prob, ptrs):
    # k_new, v_new, positions, table, k_cache, v_cache, k_scale, v_scale, status
    return lib.mfa_kv_append(ctypes.byref(prob), *ptrs, None)


def test_kv_append_validates_before_touching_the_device(lib):
    bf = problem()
    f8 = problem(kv_dtype=mfa.MFA_KV_FP8_E4M3)
    good = [0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 0x8000, 0x9000]
    for i in range(6):                       # every array but the scales and the status word
        bad = list(good); bad[i] = None
        assert _append_raw(lib, bf, bad) == mfa.MFA_ERR_INVALID_ARG
    for i, off in ((0, 8), (1, 8), (2, 2), (3, 2), (4, 8), (5, 8)):
        bad = list(good); bad[i] += off
        assert _append_raw(lib, bf, bad) == mfa.MFA_ERR_INVALID_ARG
    no_scale = list(good); no_scale[6] = None
    assert _append_raw(lib, f8, no_scale) == mfa.MFA_ERR_INVALID_ARG
    mx = problem(kv_dtype=mfa.MFA_KV_MXFP4)
    assert _append_raw(lib, mx, no_scale) == mfa.MFA_ERR_INVALID_ARG
    odd_scale = list(good); odd_scale[7] += 4   # MXFP4 writes the 8 scale bytes of a row at once
    assert _append_raw(lib, mx, odd_scale) == mfa.MFA_ERR_INVALID_ARG
    odd_status = list(good); odd_status[8] = 0x9002
    assert _append_raw(lib, f8, odd_status) == mfa.MFA_ERR_INVALID_ARG
    assert _append_raw(lib, problem(head_dim=128), good) == mfa.MFA_ERR_UNSUPPORTED
    assert _append_raw(lib, problem(head_dim=128, num_kv_heads=4), good) == mfa.MFA_ERR_UNSUPPORTED
    assert _append_raw(lib, problem(num_q_heads=128, head_dim=512, kv_shared=True), good) == mfa.MFA_ERR_UNSUPPORTED
    assert _append_raw(lib, problem(batch=-1), good) == mfa.MFA_ERR_INVALID_ARG


def test_kv_append_of_an_empty_batch_enqueues_nothing(lib):
    assert _append_raw(lib, problem(batch=0), [None] * 9) == mfa.MFA_OK


def test_run_host_validates_before_enqueuing_anything(lib):
    prob = problem()
    plan = mfa.mfa_decode_plan(prob, [10, 20, 30, 40], num_sms=8)
    P = ctypes.c_void_p
    # q_h, table_h, lens_h, out_h, lse_h, q_d, table_d, lens_d, out_d, lse_d, k, v, ks, vs, ws
    good = [0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x10000, 0x20000, 0x30000, 0x40000, 0x50000,
            0x60000, 0x70000, None, None, 0x100000]

    def call(ptrs, ws_bytes=plan.workspace_bytes, pr=prob):
        return lib.mfa_decode_run_host(ctypes.byref(plan), ctypes.byref(pr), *[P(x) if x else None for x in ptrs],
                                       ctypes.c_uint64(ws_bytes), None)
    for i in (0, 1, 2, 3, 5, 6, 7, 8, 10, 11, 14):   # every required host or device buffer
        bad = list(good); bad[i] = None
        assert call(bad) == mfa.MFA_ERR_INVALID_ARG, i
    no_lse_host = list(good); no_lse_host[4] = None     # lse on one side only
    assert call(no_lse_host) == mfa.MFA_ERR_INVALID_ARG
    odd = list(good); odd[5] = 0x10008                  # q on the device must be 16-byte aligned
    assert call(odd) == mfa.MFA_ERR_INVALID_ARG
    assert call(good, plan.workspace_bytes - 1) == mfa.MFA_ERR_WORKSPACE
    assert call(good, pr=problem(batch=5)) == mfa.MFA_ERR_INVALID_ARG


def test_decode_append_run_validates_before_touching_the_device(lib):
    """The fused append-and-decode entry point refuses bad arguments without enqueueing."""
    prob = problem()
    plan = mfa.mfa_decode_plan(prob, [10, 20, 30, 40], num_sms=8)
    P = ctypes.c_void_p
    base = [0x1000, 0x2000, 0x3000, None, None, 0x6000, 0x7000]   # q, k, v, ks, vs, table, lens
    newp = [0xA000, 0xB000, 0xC000]                               # k_new, v_new, positions
    tail = [0x8000, 0x9000, 0x10000]                               # out, lse, workspace

    def call(pr, pl, b=base, n=newp):
        return lib.mfa_decode_append_run(ctypes.byref(pl), ctypes.byref(pr), *[P(x) if x else None for x in b],
                                         *[P(x) if x else None for x in n], P(tail[0]), P(tail[1]), P(tail[2]),
                                         ctypes.c_uint64(pl.workspace_bytes), None)
    for i in range(3):
        bad = list(newp); bad[i] = None
        assert call(prob, plan, n=bad) == mfa.MFA_ERR_INVALID_ARG
    assert call(prob, plan, n=[0xA008, 0xB000, 0xC000]) == mfa.MFA_ERR_INVALID_ARG
    assert call(prob, plan, n=[0xA000, 0xB000, 0xC002]) == mfa.MFA_ERR_INVALID_ARG
    gqa = problem(head_dim=128, num_kv_heads=4)
    gplan = mfa.mfa_decode_plan(gqa, [10, 20, 30, 40], num_sms=8)
    assert call(gqa, gplan) == mfa.MFA_ERR_UNSUPPORTED
