"""Parity of the KV-cache append kernel (through the C ABI) with the oracle's append.

The bar is bit-exact: the same bf16 bits, e4m3 codes and fp32 scales, or E2M1 codes and E8M0
scale bytes, in every byte of both pools (a quantised code is an integer decided by fp32
divisions, or exact power-of-two scalings, that both sides round to nearest).  Every other slot keeps its bytes.  An append followed by a decode on the same
stream must give the oracle's attention over the oracle-appended cache.
"""
import numpy as np
import pytest
import torch

import decode_attention_02_gb300 as mfa
import oracle
from decode_attention_02_gb300 import inputs

pytestmark = pytest.mark.gpu

RAGGED = [1, 64, 65, 127, 128, 129, 200, 7, 300, 63, 2, 192, 256, 5, 66, 190, 33]


def kv_of(case):
    return mfa.KV_DTYPES[case.workload.kv_dtype]


def gpu_append(case, step, positions=None, block_table=None, status=None, tokens_per_seq=1):
    dev = "cuda"
    pr = mfa.make_problem(case.seq_lens.shape[0], case.max_pages, case.num_blocks, kv_of(case),
                          tokens_per_seq=tokens_per_seq)
    kc, vc = case.k_cache.to(dev), case.v_cache.to(dev)
    ks = None if case.k_scale is None else case.k_scale.to(dev)
    vs = None if case.v_scale is None else case.v_scale.to(dev)
    pos = (step.positions if positions is None else positions).to(dev)
    table = (case.block_table if block_table is None else block_table).to(dev)
    mfa.mfa_kv_append(pr, step.k_new.to(dev), step.v_new.to(dev), pos, table, kc, vc, ks, vs,
                      device_status=status)
    torch.cuda.synchronize()
    return kc, vc, ks, vs


def as_bits(t):
    if t is None:
        return None
    t = t.cpu()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    elif t.dtype == torch.float32:
        t = t.view(torch.int32)
    return t.numpy()


def oracle_append(case, step, positions=None, block_table=None, tokens_per_seq=1):
    return oracle.kv_append(step.k_new, step.v_new, step.positions if positions is None else positions,
                            case.block_table if block_table is None else block_table, case.k_cache, case.v_cache,
                            case.k_scale, case.v_scale, tokens_per_seq=tokens_per_seq)


def assert_pools_equal(got, want):
    kc, vc, ks, vs = (as_bits(x) for x in got)
    okc, ovc, oks, ovs = want[:4]
    view = np.int16 if okc.dtype == np.int16 else okc.dtype
    assert np.array_equal(kc, okc.view(view)), "K pool differs"
    assert np.array_equal(vc, ovc.view(view)), "V pool differs"
    if oks is not None:
        sv = np.uint8 if oks.dtype == np.uint8 else np.int32   # E8M0 bytes or fp32 bits
        assert np.array_equal(ks, oks.view(sv)), "K scales differ"
        assert np.array_equal(vs, ovs.view(sv)), "V scales differ"


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3", "mxfp4"])
def test_append_matches_oracle_bit_exactly(kv_dtype):
    case = inputs.small("append", len(RAGGED), RAGGED, kv_dtype=kv_dtype, seed=61)
    step = inputs.append_step(case, seed=62, inactive_every=5)
    want = oracle_append(case, step)
    assert want[4] == 0
    assert_pools_equal(gpu_append(case, step), want)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3", "mxfp4"])
def test_append_every_row_kind_many_times(kv_dtype):
    # 8 row kinds x 40 sequences each, every slot position of a page
    lens = [1 + (7 * b) % 256 for b in range(320)]
    case = inputs.small("kinds", len(lens), lens, kv_dtype=kv_dtype, seed=63)
    step = inputs.append_step(case, seed=64)
    assert_pools_equal(gpu_append(case, step), oracle_append(case, step))


def test_append_full_size_fp8_batch():
    w = inputs.WORKLOADS["b128_l4096_fp8"]
    case = inputs.generate(w)                      # 4096 tokens: the new one at 4095
    step = inputs.append_step(case, seed=65)
    assert_pools_equal(gpu_append(case, step), oracle_append(case, step))


def test_append_full_size_mxfp4_batch():
    case = inputs.generate(inputs.WORKLOADS["b128_l4096_mxfp4"])
    step = inputs.append_step(case, seed=75)
    assert_pools_equal(gpu_append(case, step), oracle_append(case, step))


def test_append_reports_bad_rows_and_writes_the_rest():
    case = inputs.small("bad", len(RAGGED), RAGGED, kv_dtype="fp8_e4m3", seed=66)
    step = inputs.append_step(case, seed=67)
    pos = step.positions.clone()
    table = case.block_table.clone()
    pos[0] = 64 * table.shape[1]
    t = int(pos[3])
    table[3, t // 64] = case.num_blocks
    want = oracle_append(case, step, positions=pos, block_table=table)
    assert want[4] == oracle.APPEND_BAD_BLOCK | oracle.APPEND_BAD_POSITION
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = gpu_append(case, step, positions=pos, block_table=table, status=status)
    assert_pools_equal(got, want)
    assert int(status.item()) == mfa.MFA_DEV_BAD_BLOCK | mfa.MFA_DEV_BAD_LENGTH


def test_append_without_new_tokens_changes_nothing():
    case = inputs.small("none", 5, [3, 64, 65, 130, 1], kv_dtype="fp8_e4m3", seed=68)
    step = inputs.append_step(case, seed=69)
    none = torch.full_like(step.positions, -1)
    got = gpu_append(case, step, positions=none)
    assert_pools_equal(got, (as_bits(case.k_cache).view(np.uint8), as_bits(case.v_cache).view(np.uint8),
                             case.k_scale.numpy(), case.v_scale.numpy()))


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3", "mxfp4"])
@pytest.mark.parametrize("flags", [0, mfa.MFA_PLAN_EARLY_METADATA])
def test_append_then_decode_sees_the_new_token(kv_dtype, flags):
    """One decode step: append (a programmatic dependent launch) then decode, one stream."""
    case = inputs.small("step", len(RAGGED), RAGGED, kv_dtype=kv_dtype, seed=70)
    # N(0,1) rows: values inside the decode's ranges (FP8 V scales <= 146)
    step = inputs.append_step(case, seed=71, kinds=("normal",))
    kc, vc, ks, vs, mask = oracle_append(case, step)
    assert mask == 0
    appended = inputs.Case(workload=case.workload, q=case.q,
                           k_cache=torch.from_numpy(kc).view(case.k_cache.dtype),
                           v_cache=torch.from_numpy(vc).view(case.v_cache.dtype),
                           k_scale=None if ks is None else torch.from_numpy(ks),
                           v_scale=None if vs is None else torch.from_numpy(vs),
                           block_table=case.block_table, seq_lens=case.seq_lens)
    ref_o, ref_lse = oracle.decode(appended)
    dev = "cuda"
    t = dict(q=case.q.to(dev), k=case.k_cache.to(dev), v=case.v_cache.to(dev), table=case.block_table.to(dev),
             lens=case.seq_lens.to(dev), ks=None if case.k_scale is None else case.k_scale.to(dev),
             vs=None if case.v_scale is None else case.v_scale.to(dev))
    dec = mfa.Decoder(case.q.shape[0], case.max_pages, case.num_blocks, kv_dtype=kv_of(case),
                      host_seq_lens=case.seq_lens.tolist(), flags=flags, out_dtype=mfa.MFA_OUT_FP32)
    mfa.mfa_read_device_status(dec.workspace, clear=True)
    for _ in range(3):   # repeated steps: the same append and decode again
        mfa.mfa_kv_append(dec.problem, step.k_new.to(dev), step.v_new.to(dev), step.positions.to(dev), t["table"],
                          t["k"], t["v"], t["ks"], t["vs"], device_status=dec.workspace)
        out, lse = dec(t["q"], t["k"], t["v"], t["table"], t["lens"], k_scale=t["ks"], v_scale=t["vs"])
    torch.cuda.synchronize()
    assert mfa.mfa_read_device_status(dec.workspace) == 0
    got = out.cpu().double().numpy()
    tol = (1e-2, 5e-3) if kv_dtype == "bf16" else (3e-2, 1.5e-2)
    assert np.abs(got - ref_o).max() <= tol[0]
    assert np.linalg.norm(got - ref_o) / np.linalg.norm(ref_o) <= tol[1]
    assert np.abs(lse.cpu().double().numpy() - ref_lse).max() <= 2e-3


@pytest.mark.parametrize("T", [2, 3])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3", "mxfp4"])
def test_append_of_several_tokens_matches_oracle(T, kv_dtype):
    """Multi-token step: T new rows per sequence at positions[b] .. positions[b] + T - 1, some
    across a page boundary, some sequences too short to hold T (skipped)."""
    lens = [1, 2, 64, 65, 66, 128, 130, 300, 3, 0]
    case = inputs.small("append_t", len(lens), lens, kv_dtype=kv_dtype, seed=93 + T, tokens_per_seq=T)
    step = inputs.append_step(case, seed=94, tokens_per_seq=T)
    want = oracle_append(case, step, tokens_per_seq=T)
    assert want[4] == 0
    assert_pools_equal(gpu_append(case, step, tokens_per_seq=T), want)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3", "mxfp4"])
def test_multi_token_append_then_decode(kv_dtype):
    """A multi-token step on one stream: append the T new rows, then decode the T query tokens
    (causal among them), against the oracle's decode over the oracle-appended cache."""
    T = 2
    case = inputs.small("mtp_step", len(RAGGED), RAGGED, kv_dtype=kv_dtype, seed=95, tokens_per_seq=T)
    step = inputs.append_step(case, seed=96, tokens_per_seq=T, kinds=("normal",))
    kc, vc, ks, vs, mask = oracle_append(case, step, tokens_per_seq=T)
    assert mask == 0
    appended = inputs.Case(workload=case.workload, q=case.q,
                           k_cache=torch.from_numpy(kc).view(case.k_cache.dtype),
                           v_cache=torch.from_numpy(vc).view(case.v_cache.dtype),
                           k_scale=None if ks is None else torch.from_numpy(ks),
                           v_scale=None if vs is None else torch.from_numpy(vs),
                           block_table=case.block_table, seq_lens=case.seq_lens)
    ref_o, ref_lse = oracle.decode(appended)
    dev = "cuda"
    t = dict(q=case.q.to(dev), k=case.k_cache.to(dev), v=case.v_cache.to(dev), table=case.block_table.to(dev),
             lens=case.seq_lens.to(dev), ks=None if case.k_scale is None else case.k_scale.to(dev),
             vs=None if case.v_scale is None else case.v_scale.to(dev))
    dec = mfa.Decoder(case.seq_lens.shape[0], case.max_pages, case.num_blocks, kv_dtype=kv_of(case),
                      host_seq_lens=case.seq_lens.tolist(), flags=mfa.MFA_PLAN_EARLY_METADATA,
                      out_dtype=mfa.MFA_OUT_FP32, tokens_per_seq=T)
    mfa.mfa_read_device_status(dec.workspace, clear=True)
    mfa.mfa_kv_append(dec.problem, step.k_new.to(dev), step.v_new.to(dev), step.positions.to(dev), t["table"],
                      t["k"], t["v"], t["ks"], t["vs"], device_status=dec.workspace)
    out, lse = dec(t["q"], t["k"], t["v"], t["table"], t["lens"], k_scale=t["ks"], v_scale=t["vs"])
    torch.cuda.synchronize()
    assert mfa.mfa_read_device_status(dec.workspace) == 0
    got = out.cpu().double().numpy()
    tol = (1e-2, 5e-3) if kv_dtype == "bf16" else (3e-2, 1.5e-2)
    assert np.abs(got - ref_o).max() <= tol[0]
    assert np.linalg.norm(got - ref_o) / np.linalg.norm(ref_o) <= tol[1]
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isneginf(lse.cpu().numpy()), np.isneginf(ref_lse))
    assert np.abs(lse.cpu().double().numpy()[fin] - ref_lse[fin]).max() <= 2e-3


def _fused_step(case, step, flags=0, force_ctas=0, tokens_per_seq=1, positions=None):
    """One mfa_decode_append_run on device copies of case: returns (caches, out, lse, dec)."""
    dev = "cuda"
    t = dict(q=case.q.to(dev), k=case.k_cache.to(dev), v=case.v_cache.to(dev), table=case.block_table.to(dev),
             lens=case.seq_lens.to(dev), ks=None if case.k_scale is None else case.k_scale.to(dev),
             vs=None if case.v_scale is None else case.v_scale.to(dev))
    dec = mfa.Decoder(case.seq_lens.shape[0], case.max_pages, case.num_blocks, kv_dtype=kv_of(case),
                      host_seq_lens=case.seq_lens.tolist(), flags=flags, force_ctas=force_ctas,
                      out_dtype=mfa.MFA_OUT_FP32, tokens_per_seq=tokens_per_seq)
    rows = case.q.shape[0]
    out = torch.empty((rows, 64, 256), dtype=torch.float32, device=dev)
    lse = torch.empty((rows, 64), dtype=torch.float32, device=dev)
    pos = (step.positions if positions is None else positions).to(dev)
    mfa.mfa_decode_append_run(dec.plan, dec.problem, t["q"], t["k"], t["v"], t["ks"], t["vs"], t["table"], t["lens"],
                              step.k_new.to(dev), step.v_new.to(dev), pos, out, lse, dec.workspace)
    torch.cuda.synchronize()
    return (t["k"], t["v"], t["ks"], t["vs"]), out, lse, dec


def _oracle_after_append(case, step, tokens_per_seq=1, positions=None):
    kc, vc, ks, vs, mask = oracle_append(case, step, positions=positions, tokens_per_seq=tokens_per_seq)
    appended = inputs.Case(workload=case.workload, q=case.q,
                           k_cache=torch.from_numpy(kc).view(case.k_cache.dtype),
                           v_cache=torch.from_numpy(vc).view(case.v_cache.dtype),
                           k_scale=None if ks is None else torch.from_numpy(ks),
                           v_scale=None if vs is None else torch.from_numpy(vs),
                           block_table=case.block_table, seq_lens=case.seq_lens)
    return (kc, vc, ks, vs, mask), oracle.decode(appended)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3", "mxfp4"])
@pytest.mark.parametrize("flags, force_ctas", [(0, 0), (mfa.MFA_PLAN_EARLY_METADATA, 0), (mfa.MFA_PLAN_CHECK, 7)])
def test_fused_append_decode_matches_the_oracle(kv_dtype, flags, force_ctas):
    """mfa_decode_append_run with one new token per sequence (one kernel): the caches equal the
    oracle's append byte for byte, and the decode equals the oracle's over the appended cache.
    Some sequences append no row (position -1); the others at their last position."""
    case = inputs.small("fused", len(RAGGED), RAGGED, kv_dtype=kv_dtype, seed=80)
    step = inputs.append_step(case, seed=81, inactive_every=5, kinds=("normal",))
    want, (ref_o, ref_lse) = _oracle_after_append(case, step)
    assert want[4] == 0
    caches, out, lse, dec = _fused_step(case, step, flags=flags, force_ctas=force_ctas)
    assert_pools_equal(caches, want)
    assert mfa.mfa_read_device_status(dec.workspace) == 0
    got = out.cpu().double().numpy()
    tol = (1e-2, 5e-3) if kv_dtype == "bf16" else (3e-2, 1.5e-2)
    assert np.abs(got - ref_o).max() <= tol[0]
    assert np.linalg.norm(got - ref_o) / np.linalg.norm(ref_o) <= tol[1]
    assert np.abs(lse.cpu().double().numpy() - ref_lse).max() <= 2e-3


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3", "mxfp4"])
def test_fused_append_writes_rows_past_the_length_and_reports_bad_ones(kv_dtype):
    """Rows at or past a sequence's length (read by nobody this step) are written as well; a
    position past the block table and a page id outside the pool are reported and skipped,
    exactly as by the append kernel."""
    case = inputs.small("fused_past", len(RAGGED), RAGGED, kv_dtype=kv_dtype, seed=82)
    step = inputs.append_step(case, seed=83, kinds=("normal",))
    pos = step.positions.clone()
    lens = case.seq_lens
    for b in (1, 4, 9):           # one past the last token, inside the same page
        if int(lens[b]) % 64 != 0:
            pos[b] = int(lens[b])
    pos[6] = 64 * case.block_table.shape[1]          # past the table: BAD_LENGTH
    table = case.block_table.clone()
    table[11, int(pos[11]) // 64] = case.num_blocks   # outside the pool: BAD_BLOCK
    bad = inputs.Case(workload=case.workload, q=case.q, k_cache=case.k_cache, v_cache=case.v_cache,
                      k_scale=case.k_scale, v_scale=case.v_scale, block_table=table, seq_lens=case.seq_lens)
    want, _ = _oracle_after_append(bad, step, positions=pos)
    assert want[4] == oracle.APPEND_BAD_BLOCK | oracle.APPEND_BAD_POSITION
    caches, out, lse, dec = _fused_step(bad, step, positions=pos)
    assert_pools_equal(caches, want)
    st = mfa.mfa_read_device_status(dec.workspace)
    assert st & mfa.MFA_DEV_BAD_LENGTH and st & mfa.MFA_DEV_BAD_BLOCK


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_fused_append_with_several_tokens_runs_the_two_kernels(kv_dtype):
    """T = 2: the append kernel first, then the decode; the same bytes and bits as the two
    separate calls."""
    T = 2
    case = inputs.small("fused_t2", len(RAGGED), RAGGED, kv_dtype=kv_dtype, seed=84, tokens_per_seq=T)
    step = inputs.append_step(case, seed=85, tokens_per_seq=T, kinds=("normal",))
    caches, out, lse, dec = _fused_step(case, step, tokens_per_seq=T)
    kc, vc, ks, vs = gpu_append(case, step, tokens_per_seq=T)
    assert_pools_equal(caches, tuple(as_bits(x) for x in (kc, vc, ks, vs)) + (0,))
    dev = "cuda"
    out2, lse2 = dec(case.q.to(dev), kc, vc, case.block_table.to(dev), case.seq_lens.to(dev), k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert torch.equal(out2.view(torch.int32), out.view(torch.int32))
    assert torch.equal(lse2, lse)
