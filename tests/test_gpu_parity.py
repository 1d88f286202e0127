"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Limits (stated for the MFA decode step): bf16 KV max-abs <= 1e-2 and
relative-L2 <= 5e-3; block-table and length indexing exact (NaN-poisoned
unused slots and pages must not reach the output).  lse is compared to 2e-3
absolute.  The limits apply to the kernel's fp32 result (the fp32 output
mode).  The bf16 output is checked to be exactly the round-to-nearest-even of
that fp32 result, and against the oracle with half a bf16 ulp (<= 2^-8 |r|)
added to the max-abs limit: a bf16 output cannot be closer than that.
"""
import numpy as np
import pytest
import torch

import decode_attention_02_gb300 as mfa
import oracle
from decode_attention_02_gb300 import inputs

pytestmark = pytest.mark.gpu

BF16_MAX_ABS, BF16_REL_L2 = 1e-2, 5e-3
LSE_ABS = 2e-3


def to_dev(case, dev="cuda"):
    return dict(q=case.q.to(dev), k_cache=case.k_cache.to(dev), v_cache=case.v_cache.to(dev),
                block_table=case.block_table.to(dev), seq_lens=case.seq_lens.to(dev),
                k_scale=None if case.k_scale is None else case.k_scale.to(dev),
                v_scale=None if case.v_scale is None else case.v_scale.to(dev))


def shape_of(w):
    """The library shape tuple of a workload (query heads, head width, key/value heads, shared)."""
    return (w.num_q_heads, w.head_dim, w.num_kv_heads, w.kv_shared)


def gpu_decode(case, force_ctas=0, flags=mfa.MFA_PLAN_CHECK, stream=None, out_dtype=mfa.MFA_OUT_FP32):
    t = to_dev(case)
    w = case.workload
    kv = mfa.KV_DTYPES[w.kv_dtype]
    dec = mfa.Decoder(case.seq_lens.shape[0],
                      case.max_pages, case.num_blocks, kv_dtype=kv,
                      softmax_scale=w.scale(), host_seq_lens=case.seq_lens.tolist(),
                      force_ctas=force_ctas, flags=flags, out_dtype=out_dtype, tokens_per_seq=w.tokens_per_seq,
                      shape=shape_of(w))
    out, lse = dec(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"],
                   k_scale=t["k_scale"], v_scale=t["v_scale"], stream=stream)
    torch.cuda.synchronize()
    return out, lse, dec


def check_parity(case, out, lse, max_abs=BF16_MAX_ABS, rel_l2=BF16_REL_L2, ref=None):
    ref_o, ref_lse = oracle.decode(case) if ref is None else ref
    got = out.float().cpu().double().numpy()
    assert np.all(np.isfinite(got)), "non-finite output"
    err = np.abs(got - ref_o)
    denom = np.linalg.norm(ref_o)
    rel = np.linalg.norm(got - ref_o) / denom if denom > 0 else np.linalg.norm(got - ref_o)
    # bf16 outputs may sit half an ulp (<= 2^-8 |r|) from the exact value
    allow = max_abs + (np.abs(ref_o) * 2.0 ** -8 if out.dtype == torch.bfloat16 else 0.0)
    assert np.all(err <= allow), f"max-abs {err.max():.3e} (beyond rounding: {(err - allow).max():.3e})"
    assert rel <= rel_l2, f"rel-L2 {rel:.3e}"
    g_lse = lse.cpu().double().numpy()
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isneginf(g_lse), np.isneginf(ref_lse))
    if fin.any():
        assert np.abs(g_lse[fin] - ref_lse[fin]).max() <= LSE_ABS, "lse mismatch"
    return err.max(initial=0.0), rel


def test_tiny_workload_matches_oracle():
    case = inputs.generate(inputs.WORKLOADS["tiny_b1_l512_bf16"])
    out, lse, _ = gpu_decode(case)
    check_parity(case, out, lse)


RAGGED_LENS = [1, 63, 64, 65, 127, 128, 129, 200, 0, 517, 1000, 300]


@pytest.mark.parametrize("force_ctas", [0, 1, 2, 3, 7, 16, 64])
def test_ragged_lengths_any_split(force_ctas):
    case = inputs.small("ragged", len(RAGGED_LENS), RAGGED_LENS, seed=7, extra_blocks=3)
    out, lse, _ = gpu_decode(case, force_ctas=force_ctas)
    check_parity(case, out, lse)


def test_spiked_keys():
    case = inputs.small("spike", 6, [1024, 2000, 1500, 777, 4096, 3000], seed=8, k_spike_frac=0.01)
    out, lse, _ = gpu_decode(case)
    check_parity(case, out, lse)


def test_length_one_returns_v0_bit_exactly():
    case = inputs.small("l1", 3, [1, 1, 1], seed=9)
    out, lse, _ = gpu_decode(case, out_dtype=mfa.MFA_OUT_BF16)
    for b in range(3):
        blk = int(case.block_table[b, 0])
        v0 = case.v_cache[blk, 0]
        assert torch.equal(out[b].cpu().view(torch.int16), v0.expand(64, -1).view(torch.int16))


def test_block_permutation_is_bitwise_invariant():
    case = inputs.small("perm", 5, [100, 640, 1, 333, 2049], seed=10, extra_blocks=4)
    out1, lse1, _ = gpu_decode(case, force_ctas=5, out_dtype=mfa.MFA_OUT_BF16)
    nb = case.num_blocks
    perm = torch.from_numpy(np.random.default_rng(1).permutation(nb))
    k2 = torch.empty_like(case.k_cache); k2[perm] = case.k_cache
    v2 = torch.empty_like(case.v_cache); v2[perm] = case.v_cache
    table = case.block_table.clone()
    used = table >= 0
    table[used] = perm[table[used].long()].to(torch.int32)
    case2 = inputs.Case(case.workload, case.q, k2, v2, None, None, table, case.seq_lens)
    out2, lse2, _ = gpu_decode(case2, force_ctas=5, out_dtype=mfa.MFA_OUT_BF16)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)


def test_constant_keys_give_mean_of_values():
    case = inputs.small("constk", 2, [300, 1000], seed=11)
    for b in range(2):
        row = case.k_cache[int(case.block_table[b, 0]), 0].clone()
        L = int(case.seq_lens[b])
        for t in range(L):
            case.k_cache[int(case.block_table[b, t // 64]), t % 64] = row
    out, lse, _ = gpu_decode(case, force_ctas=3)
    for b in range(2):
        L = int(case.seq_lens[b])
        t = np.arange(L)
        V = case.v_cache[case.block_table[b, t // 64].long(), torch.from_numpy(t % 64)].double()
        mean = V.mean(dim=0)
        assert (out[b].cpu().double() - mean[None]).abs().max() <= BF16_MAX_ABS


def test_empty_sequences_give_zero_and_minus_inf():
    case = inputs.small("empty", 4, [0, 70, 0, 0], seed=12)
    for fc in (0, 1, 3):
        out, lse, _ = gpu_decode(case, force_ctas=fc)
        assert torch.all(out[[0, 2, 3]] == 0)
        assert torch.all(torch.isneginf(lse[[0, 2, 3]]))
        check_parity(case, out, lse)


def test_all_empty_batch():
    case = inputs.small("allempty", 3, [0, 0, 0], seed=13)
    out, lse, _ = gpu_decode(case)
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_separate_combine_matches_fused_run():
    case = inputs.small("sep", 4, [900, 1, 2500, 64], seed=14)
    out1, lse1, _ = gpu_decode(case, force_ctas=9, out_dtype=mfa.MFA_OUT_BF16)
    t = to_dev(case)
    dec = mfa.Decoder(4, case.max_pages, case.num_blocks, host_seq_lens=case.seq_lens.tolist(), force_ctas=9,
                      flags=mfa.MFA_PLAN_NO_COMBINE)
    out2 = torch.empty_like(out1)
    lse2 = torch.empty_like(lse1)
    dec(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"], out=out2, lse=lse2)
    mfa.mfa_combine(dec.plan, dec.problem, dec.workspace, t["seq_lens"], out2, lse2)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)


@pytest.mark.parametrize("kv", [mfa.MFA_KV_BF16, mfa.MFA_KV_FP8_E4M3])
def test_combine_kernel_against_oracle_merge(kv):
    """mfa_combine alone on random partials laid out as include/mfa.h documents."""
    lens = [129, 1000, 5, 640]
    B, G = len(lens), 6
    prob = mfa.make_problem(B, 16, 64, kv)
    plan = mfa.mfa_decode_plan(prob, lens, force_ctas=G, num_sms=152)
    ws = torch.zeros(int(plan.workspace_bytes), dtype=torch.uint8, device="cuda")
    o_off, l_off = mfa.workspace_layout(plan)
    S = plan.num_partials
    g = torch.Generator().manual_seed(0)
    po = torch.randn(S, 64, 256, generator=g)
    pl = torch.randn(S, 64, generator=g) * 3
    ws[o_off:o_off + po.numel() * 4] = po.view(torch.uint8).reshape(-1).cuda()
    ws[l_off:l_off + pl.numel() * 4] = pl.view(torch.uint8).reshape(-1).cuda()
    out = torch.zeros(B, 64, 256, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(B, 64, device="cuda")
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    assert prob.out_dtype == mfa.MFA_OUT_BF16
    mfa.mfa_combine(plan, prob, ws, seq, out, lse)
    torch.cuda.synchronize()
    # the documented split: tile k of sequence b at cost 4 (S_b + k) + c N_b; CTA g owns
    # costs [floor(g C / G), floor((g + 1) C / G)), C = 4 W + c (N - 1); c = 3 (bf16 KV) or 10
    c = 10 if kv == mfa.MFA_KV_FP8_E4M3 else 3
    tiles = [(L + 127) // 128 for L in lens]
    W, N = sum(tiles), sum(1 for t in tiles if t > 0)
    C = 4 * W + c * max(N - 1, 0)
    before = nonempty = 0
    for b in range(B):
        base = 4 * before + c * nonempty
        costs = [base + 4 * k for k in range(tiles[b])]
        covering = sorted({max(gg for gg in range(G) if (gg * C) // G <= c) for c in costs})
        before += tiles[b]
        nonempty += tiles[b] > 0
        if len(covering) < 2:
            continue   # written by the decode kernel, not by combine
        slots = [b + gg for gg in covering]
        ro, rl = oracle.combine(po[slots].double().numpy(), pl[slots].double().numpy())
        assert np.abs(out[b].cpu().double().numpy() - ro).max() <= 1e-2 + 1e-2 * np.abs(ro).max()
        assert np.abs(lse[b].cpu().double().numpy() - rl).max() <= 1e-4


def test_bad_block_id_is_reported_not_faulted():
    case = inputs.small("badblk", 2, [100, 200], seed=15)
    case.block_table[1, 2] = case.num_blocks + 7
    with pytest.raises(mfa.MfaError) as e:
        gpu_decode(case)
    assert e.value.status == mfa.MFA_ERR_DEVICE_CHECK


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3", "mxfp4"])
@pytest.mark.parametrize("bad_id", [-3, 10 ** 6])
def test_bad_block_id_reads_as_a_page_of_zeros(kv, bad_id):
    """A block id outside the pool is reported, and its page contributes zero keys and zero
    values: the output equals the oracle's over a cache whose entry points at a zero page."""
    case = inputs.small("badblk0", 3, [100, 200, 150], kv_dtype=kv, seed=15)
    ref_case = inputs.small("badblk0", 3, [100, 200, 150], kv_dtype=kv, seed=15)
    case.block_table[1, 2] = bad_id
    # the oracle's input: one more physical page, all zeros (e4m3 code 0 with scale 1)
    nb = ref_case.num_blocks
    zero_k = torch.zeros((1,) + tuple(ref_case.k_cache.shape[1:]), dtype=ref_case.k_cache.dtype)
    ref_case.k_cache = torch.cat([ref_case.k_cache, zero_k]).contiguous()
    ref_case.v_cache = torch.cat([ref_case.v_cache, zero_k.clone()]).contiguous()
    if ref_case.k_scale is not None and kv == "mxfp4":
        one = torch.full((1,) + tuple(ref_case.k_scale.shape[1:]), 127, dtype=torch.uint8)   # E8M0 1.0
        ref_case.k_scale = torch.cat([ref_case.k_scale, one]).contiguous()
        ref_case.v_scale = torch.cat([ref_case.v_scale, one.clone()]).contiguous()
    elif ref_case.k_scale is not None:
        one = torch.ones((1, ref_case.k_scale.shape[1]), dtype=torch.float32)
        ref_case.k_scale = torch.cat([ref_case.k_scale, one]).contiguous()
        ref_case.v_scale = torch.cat([ref_case.v_scale, one.clone()]).contiguous()
    ref_case.block_table[1, 2] = nb
    out, lse, dec = gpu_decode(case, flags=0)
    assert mfa.mfa_read_device_status(dec.workspace) == mfa.MFA_DEV_BAD_BLOCK
    lim = (BF16_MAX_ABS, BF16_REL_L2) if kv == "bf16" else (3e-2, 1.5e-2)
    check_parity(case, out, lse, *lim, ref=oracle.decode(ref_case))


def test_length_beyond_table_is_reported():
    case = inputs.small("badlen", 2, [100, 200], seed=16)
    t = to_dev(case)
    dec = mfa.Decoder(2, case.max_pages, case.num_blocks, max_seq_len=case.max_pages * 64,
                      flags=mfa.MFA_PLAN_CHECK)
    t["seq_lens"][1] = case.max_pages * 64 + 1
    with pytest.raises(mfa.MfaError) as e:
        dec(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"])
    assert e.value.status == mfa.MFA_ERR_DEVICE_CHECK
    assert mfa.mfa_read_device_status(dec.workspace) & mfa.MFA_DEV_BAD_LENGTH


def test_early_metadata_chain_matches():
    """Back-to-back steps with MFA_PLAN_EARLY_METADATA (decode launched as a programmatic
    dependent of the previous step's combine) give the same bits as plain steps."""
    case = inputs.small("pdl", 6, [4096, 1000, 64, 2500, 1, 3000], seed=19)
    ref16, refl, _ = gpu_decode(case, out_dtype=mfa.MFA_OUT_BF16)
    t = to_dev(case)
    dec = mfa.Decoder(6, case.max_pages, case.num_blocks, host_seq_lens=case.seq_lens.tolist(),
                      flags=mfa.MFA_PLAN_EARLY_METADATA)
    outs = []
    for _ in range(4):
        o, l = dec(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"])
        outs.append((o, l))
    torch.cuda.synchronize()
    assert mfa.mfa_read_device_status(dec.workspace) == 0
    for o, l in outs:
        assert torch.equal(o.view(torch.int16), ref16.view(torch.int16))
        assert torch.equal(l, refl)


def test_runs_on_a_side_stream():
    case = inputs.small("stream", 3, [700, 50, 1300], seed=17)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out, lse, _ = gpu_decode(case, stream=s)
    check_parity(case, out, lse)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("force_ctas", [1, 2, 5, 9, 13, 14, 15, 17])
def test_cost_balanced_split_with_empty_runs(kv_dtype, force_ctas):
    # 13 tiles over sequences with runs of empties: CTA ranges fall on sequence boundaries,
    # inside boundary costs and (beyond 13 CTAs) on nothing at all; decode and combine must
    # agree on which CTA holds which tiles
    lens = [0, 0, 129, 0, 1, 256, 0, 0, 700, 64, 0, 65, 0]
    case = inputs.small("cost", len(lens), lens, kv_dtype=kv_dtype, seed=79)
    out, lse, dec = gpu_decode(case, force_ctas=force_ctas)
    limits = dict(max_abs=3e-2, rel_l2=1.5e-2) if kv_dtype != "bf16" else {}
    check_parity(case, out, lse, **limits)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_batch_larger_than_one_thread_per_sequence(kv_dtype):
    # more sequences than the decode kernel has threads: the schedule takes its chunked path
    rng = np.random.default_rng(77)
    lens = [int(x) for x in rng.integers(0, 300, size=600)]
    lens[5] = 0
    lens[599] = 257
    case = inputs.small("bigb", len(lens), lens, kv_dtype=kv_dtype, seed=78)
    out, lse, dec = gpu_decode(case)
    limits = dict(max_abs=3e-2, rel_l2=1.5e-2) if kv_dtype != "bf16" else {}
    check_parity(case, out, lse, **limits)


@pytest.mark.parametrize("name", ["b32_l4096_bf16", "ragged_b128_l1024_8192_bf16", "long_b4_l131072_bf16"])
def test_full_size_workload(name):
    """Full-size workloads in the launch configuration the benchmark times."""
    case = inputs.generate(inputs.WORKLOADS[name])
    out, lse, dec = gpu_decode(case)
    assert dec.plan.num_ctas == min(torch.cuda.get_device_properties(0).multi_processor_count,
                                    int(dec.plan.total_tiles))
    ref = oracle.decode(case)
    check_parity(case, out, lse, ref=ref)
    out16, lse16, _ = gpu_decode(case, out_dtype=mfa.MFA_OUT_BF16)
    assert torch.equal(out16.view(torch.int16), out.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(lse16, lse)
    check_parity(case, out16, lse16, ref=ref)


@pytest.mark.parametrize("force_ctas", [0, 1, 5, 40])
def test_bf16_output_is_rne_of_fp32_output(force_ctas):
    case = inputs.small("rne", 5, [3000, 64, 1, 700, 1500], seed=18, k_spike_frac=0.01)
    o32, l32, _ = gpu_decode(case, force_ctas=force_ctas)
    o16, l16, _ = gpu_decode(case, force_ctas=force_ctas, out_dtype=mfa.MFA_OUT_BF16)
    assert torch.equal(o16.view(torch.int16), o32.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(l16, l32)
    ref = oracle.decode(case)
    check_parity(case, o32, l32, ref=ref)
    check_parity(case, o16, l16, ref=ref)


@pytest.mark.parametrize("name", ["ragged_b128_l1024_8192_bf16", "b128_l4096_fp8", "long_b4_l131072_fp8"])
def test_repeated_steps_are_bitwise_identical(name):
    """The split is fixed and every reduction has a fixed order, so repeated steps must give
    the same bits.  The warp roles hand tiles to one another through barriers and counts in
    shared memory; a race there shows up as a step that differs.  Twenty back-to-back steps
    on the same inputs, through the early-metadata chain the benchmark times."""
    case = inputs.generate(inputs.WORKLOADS[name])
    t = to_dev(case)
    kv = mfa.MFA_KV_FP8_E4M3 if case.workload.kv_dtype == "fp8_e4m3" else mfa.MFA_KV_BF16
    dec = mfa.Decoder(case.q.shape[0], case.max_pages, case.num_blocks, kv_dtype=kv,
                      softmax_scale=case.workload.scale(), host_seq_lens=case.seq_lens.tolist(),
                      flags=mfa.MFA_PLAN_EARLY_METADATA, out_dtype=mfa.MFA_OUT_FP32)
    mfa.mfa_read_device_status(dec.workspace, clear=True)
    outs = []
    for _ in range(20):
        out, lse = dec(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"],
                       k_scale=t["k_scale"], v_scale=t["v_scale"])
        outs.append((out.clone(), lse.clone()))
    torch.cuda.synchronize()
    assert mfa.mfa_read_device_status(dec.workspace) == 0
    o0, l0 = outs[0]
    for o, l in outs[1:]:
        assert torch.equal(o.view(torch.int32), o0.view(torch.int32))
        assert torch.equal(l.view(torch.int32), l0.view(torch.int32))
    # and the first of them is the right answer on a sample of sequences
    sample = slice(0, min(8, case.q.shape[0]))
    ref_o, ref_lse = oracle.decode(case, batch_slice=sample)
    got = o0[sample].cpu().double().numpy()
    tol = 1e-2 if kv == mfa.MFA_KV_BF16 else 3e-2
    assert np.abs(got - ref_o).max() <= tol


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_host_buffer_steps_on_two_streams_match_the_device_path(kv_dtype):
    """mfa_decode_run_host: pinned host q, table and lengths in, pinned host out and lse back,
    with two streams alternating (each with its own staging buffers and workspace, so one
    step's copies overlap the other's kernels).  Every step must give the device path's bits."""
    case = inputs.small("host", 9, [1, 64, 65, 300, 2000, 0, 129, 700, 4096], kv_dtype=kv_dtype, seed=72)
    ref_out, ref_lse, _ = gpu_decode(case, flags=0, out_dtype=mfa.MFA_OUT_BF16)
    t = to_dev(case)
    kv = mfa.MFA_KV_FP8_E4M3 if kv_dtype == "fp8_e4m3" else mfa.MFA_KV_BF16
    lanes = []
    for _ in range(2):
        dec = mfa.Decoder(case.q.shape[0], case.max_pages, case.num_blocks, kv_dtype=kv,
                          softmax_scale=case.workload.scale(), host_seq_lens=case.seq_lens.tolist(),
                          flags=mfa.MFA_PLAN_EARLY_METADATA)
        lanes.append((dec, torch.cuda.Stream()))
    q_h, table_h, lens_h = case.q.pin_memory(), case.block_table.pin_memory(), case.seq_lens.pin_memory()
    outs = [(torch.empty(ref_out.shape, dtype=torch.bfloat16).pin_memory(),
             torch.empty(ref_lse.shape, dtype=torch.float32).pin_memory()) for _ in range(6)]
    torch.cuda.synchronize()
    for i, (o_h, l_h) in enumerate(outs):
        dec, st = lanes[i % 2]
        dec.run_host(q_h, table_h, lens_h, o_h, l_h, t["k_cache"], t["v_cache"], t["k_scale"], t["v_scale"],
                     stream=st)
    torch.cuda.synchronize()
    for o_h, l_h in outs:
        assert torch.equal(o_h.view(torch.int16), ref_out.cpu().view(torch.int16))
        assert torch.equal(l_h, ref_lse.cpu())


def gpu_decode_mtp(case, force_ctas=0, out_dtype=mfa.MFA_OUT_FP32, flags=mfa.MFA_PLAN_CHECK):
    t = to_dev(case)
    kv = mfa.MFA_KV_FP8_E4M3 if case.workload.kv_dtype == "fp8_e4m3" else mfa.MFA_KV_BF16
    T = case.workload.tokens_per_seq
    dec = mfa.Decoder(case.seq_lens.shape[0], case.max_pages, case.num_blocks, kv_dtype=kv,
                      softmax_scale=case.workload.scale(), host_seq_lens=case.seq_lens.tolist(),
                      force_ctas=force_ctas, flags=flags, out_dtype=out_dtype, tokens_per_seq=T)
    out, lse = dec(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"],
                   k_scale=t["k_scale"], v_scale=t["v_scale"])
    torch.cuda.synchronize()
    return out, lse, dec


@pytest.mark.parametrize("T", [2, 3, 4])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("force_ctas", [0, 1, 7])
def test_multi_token_decode(T, kv_dtype, force_ctas):
    """T new query tokens per sequence, causal among themselves: lengths below T leave some
    query tokens with nothing to attend to (out 0, lse -inf)."""
    lens = [1, 2, 3, 0, 64, 65, 130, 257, 700, 4]
    case = inputs.small("mtp", len(lens), lens, kv_dtype=kv_dtype, seed=80 + T, tokens_per_seq=T)
    out, lse, dec = gpu_decode_mtp(case, force_ctas=force_ctas)
    assert out.shape[0] == len(lens) * T
    if kv_dtype == "bf16":
        check_parity(case, out, lse)
    else:
        check_parity(case, out, lse, max_abs=3e-2, rel_l2=1.5e-2)


@pytest.mark.parametrize("name", ["mtp2_b32_l4096_bf16", "mtp2_b32_l4096_fp8"])
def test_multi_token_decode_full_size(name):
    """Two new tokens for each of 32 sequences of 4096 (bf16 and e4m3 caches): the multi-token
    workloads, checked on a sample of sequences (the oracle runs per (sequence, token) pair)
    plus two sequences from the far end of the batch."""
    case = inputs.generate(inputs.WORKLOADS[name])
    out, lse, dec = gpu_decode_mtp(case, flags=mfa.MFA_PLAN_CHECK | mfa.MFA_PLAN_EARLY_METADATA)
    assert mfa.mfa_read_device_status(dec.workspace) == 0
    max_abs, rel_l2 = (3e-2, 1.5e-2) if name.endswith("fp8") else (BF16_MAX_ABS, BF16_REL_L2)
    for sample in (slice(0, 8), slice(60, 64)):   # pairs (sequence, token)
        ref_o, ref_lse = oracle.decode(case, batch_slice=sample)
        got = out[sample].cpu().double().numpy()
        err = np.abs(got - ref_o)
        assert err.max() <= max_abs
        assert np.linalg.norm(got - ref_o) / np.linalg.norm(ref_o) <= rel_l2
        assert np.abs(lse[sample].cpu().double().numpy() - ref_lse).max() <= LSE_ABS


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_multi_token_decode_beyond_one_thread_per_pair(kv_dtype):
    """150 sequences x 3 query tokens = 450 (sequence, token) pairs: more than the bf16 kernel's
    352 threads, so its schedule takes the chunked path (e4m3, 512 threads, the per-thread one)."""
    rng = np.random.default_rng(97)
    lens = [int(x) for x in rng.integers(0, 200, size=150)]
    case = inputs.small("mtp_many", len(lens), lens, kv_dtype=kv_dtype, seed=98, tokens_per_seq=3)
    out, lse, dec = gpu_decode_mtp(case)
    if kv_dtype == "bf16":
        check_parity(case, out, lse)
    else:
        check_parity(case, out, lse, max_abs=3e-2, rel_l2=1.5e-2)


@pytest.mark.parametrize("out_dtype", [mfa.MFA_OUT_FP32, mfa.MFA_OUT_BF16])
def test_combine_with_sixteen_heads_a_cta(out_dtype):
    """96 sequences over 152 CTAs: the combine takes 16 heads a CTA in four rounds, and with all
    of a sequence's partials in one pass it loads every round's partials together.  Lengths
    from 1 to 1,500 leave sequences whole, split in two and split over several CTAs."""
    rng = np.random.default_rng(123)
    lens = [int(x) for x in rng.integers(1, 1500, size=96)]
    lens[:4] = [1, 128, 129, 1499]
    case = inputs.small("combine16", len(lens), lens, seed=124)
    out, lse, dec = gpu_decode(case, force_ctas=152, out_dtype=out_dtype)
    assert 96 * 64 >= 16 * 2 * 152          # the host picks 16 heads a combine CTA here
    check_parity(case, out, lse)


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_ctas_without_tiles_leave_the_partials_alone(kv):
    """With 16 CTAs over these lengths, CTA 11's cost range holds no tile while sequence 0 is
    split over CTAs 0..3 (its partial from CTA 0 sits in slot 0).  A CTA without a segment
    writes nothing; repeated steps stay exact against the oracle and set no status bit."""
    lens = [700, 1, 1, 1, 1, 1, 1, 1, 1, 1, 300]
    case = inputs.small("empty_cta", len(lens), lens, kv_dtype=kv, seed=70)
    ref = oracle.decode(case)
    lim = (3e-2, 1.5e-2) if kv == "fp8_e4m3" else (BF16_MAX_ABS, BF16_REL_L2)
    for _ in range(5):
        out, lse, _ = gpu_decode(case, force_ctas=16)
        check_parity(case, out, lse, *lim, ref=ref)
