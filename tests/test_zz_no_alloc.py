"""The workspace-free decode entry point gives the same results as the regular one.

mfa_decode_run_static_workspace serves callers that cannot allocate device
memory themselves (for instance a plugin whose host application owns every
device allocation, or a latency-critical path that must not pay cudaMalloc's
implicit synchronisation): it uses a fixed scratch array that lives inside the
library.  These checks call it through the C ABI twice in a row, on two
different batches, and compare each result with mfa_decode_run's under the
limits the parity tests use, for a bf16 and an e4m3 cache and with the plan
flags the regular path takes.  The file is named so that pytest collects it
last.
"""
import numpy as np
import pytest
import torch

import decode_attention_02_gb300 as mfa
from decode_attention_02_gb300 import inputs

pytestmark = pytest.mark.gpu

# (max-abs, rel-L2, lse) of the parity tests, per KV format
LIMITS = {"bf16": (1e-2, 5e-3, 2e-3), "fp8_e4m3": (3e-2, 1.5e-2, 2e-3)}


def _device(case):
    d = "cuda"
    ks = None if case.k_scale is None else case.k_scale.to(d)
    vs = None if case.v_scale is None else case.v_scale.to(d)
    return (case.q.to(d), case.k_cache.to(d), case.v_cache.to(d), ks, vs, case.block_table.to(d),
            case.seq_lens.to(d))


def _close(a, b, max_abs, rel_l2):
    a = a.float().cpu().double().numpy()
    b = b.float().cpu().double().numpy()
    err = np.abs(a - b)
    allow = max_abs + np.abs(b) * 2.0 ** -8          # both outputs are bf16
    rel = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
    return bool(np.all(err <= allow)) and rel <= rel_l2


def _cases(kv):
    return [inputs.small("noalloc_a", 7, [4096, 1000, 64, 2500, 1, 3000, 0], kv_dtype=kv, seed=31,
                         k_spike_frac=0.01),
            inputs.small("noalloc_b", 3, [129, 700, 8000], kv_dtype=kv, seed=32)]


@pytest.mark.parametrize("kv,flags", [
    ("bf16", 0),
    ("fp8_e4m3", 0),
    ("bf16", mfa.MFA_PLAN_CHECK),
    ("fp8_e4m3", mfa.MFA_PLAN_EARLY_METADATA),
    ("bf16", mfa.MFA_PLAN_EARLY_METADATA | mfa.MFA_PLAN_CHECK),
])
def test_static_workspace_matches_regular_entry_point_on_two_calls_in_a_row(kv, flags):
    max_abs, rel_l2, lse_abs = LIMITS[kv]
    kvd = mfa.MFA_KV_FP8_E4M3 if kv == "fp8_e4m3" else mfa.MFA_KV_BF16
    for case in _cases(kv):
        q, k, v, ks, vs, table, lens = _device(case)
        B = case.q.shape[0]
        # regular entry point, workspace from PyTorch
        dec = mfa.Decoder(B, case.max_pages, case.num_blocks, kv_dtype=kvd, host_seq_lens=case.seq_lens.tolist(),
                          flags=flags)
        out_r, lse_r = dec(q, k, v, table, lens, k_scale=ks, v_scale=vs)
        # workspace-free entry point: same plan and problem, no workspace argument
        out_s = torch.full_like(out_r, float("nan"))
        lse_s = torch.full_like(lse_r, float("nan"))
        mfa.mfa_decode_run_static_workspace(dec.plan, dec.problem, q, k, v, ks, vs, table, lens, out_s, lse_s)
        torch.cuda.synchronize()
        assert dec.plan.workspace_bytes <= mfa.MFA_STATIC_WORKSPACE_BYTES
        assert torch.isfinite(out_s.float()).all()
        assert _close(out_s, out_r, max_abs, rel_l2)
        fin = torch.isfinite(lse_r)
        assert torch.equal(fin, torch.isfinite(lse_s))
        assert (lse_s[fin] - lse_r[fin]).abs().max().item() <= lse_abs


def test_static_workspace_rejects_plans_that_do_not_fit():
    B = 400
    prob = mfa.make_problem(B, 1, 4)
    plan = mfa.mfa_decode_plan(prob, None, max_seq_len=64, num_sms=152)
    assert plan.workspace_bytes > mfa.MFA_STATIC_WORKSPACE_BYTES
    small = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(mfa.MfaError) as e:
        mfa.mfa_decode_run_static_workspace(plan, prob, small, small, small, None, None, small, small, small, None)
    assert e.value.status == mfa.MFA_ERR_WORKSPACE


def test_static_workspace_rejects_a_split_plan_without_the_combine():
    """Partials left in the library's array could never reach mfa_combine: refused, and the
    call enqueues nothing (the output keeps its contents)."""
    case = inputs.small("noalloc_nc", 2, [700, 300], seed=33)
    q, k, v, ks, vs, table, lens = _device(case)
    dec = mfa.Decoder(2, case.max_pages, case.num_blocks, host_seq_lens=case.seq_lens.tolist(), force_ctas=4,
                      flags=mfa.MFA_PLAN_NO_COMBINE)
    assert dec.plan.num_ctas > 1
    out = torch.full((2, 64, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mfa.MfaError) as e:
        mfa.mfa_decode_run_static_workspace(dec.plan, dec.problem, q, k, v, ks, vs, table, lens, out, None)
    assert e.value.status == mfa.MFA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
    # a single-CTA plan has no partials: NO_COMBINE is harmless there and runs
    one = mfa.Decoder(2, case.max_pages, case.num_blocks, host_seq_lens=case.seq_lens.tolist(), force_ctas=1,
                      flags=mfa.MFA_PLAN_NO_COMBINE)
    ref, _ = mfa.Decoder(2, case.max_pages, case.num_blocks, host_seq_lens=case.seq_lens.tolist())(q, k, v, table,
                                                                                                   lens)
    mfa.mfa_decode_run_static_workspace(one.plan, one.problem, q, k, v, ks, vs, table, lens, out, None)
    torch.cuda.synchronize()
    assert _close(out, ref, *LIMITS["bf16"][:2])


def test_static_workspace_rejects_bad_arguments_before_enqueueing():
    """A misaligned q is refused before the status-word clear is enqueued."""
    case = inputs.small("noalloc_bad", 1, [100], seed=34)
    q, k, v, ks, vs, table, lens = _device(case)
    dec = mfa.Decoder(1, case.max_pages, case.num_blocks, host_seq_lens=[100])
    out = torch.empty((1, 64, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mfa.MfaError) as e:
        mfa.mfa_decode_run_static_workspace(dec.plan, dec.problem, q.data_ptr() + 2, k, v, ks, vs, table, lens, out,
                                            None)
    assert e.value.status == mfa.MFA_ERR_INVALID_ARG


def test_static_workspace_device_checks_surface_through_plan_check():
    """The array's status word is private: a block id outside the pool is reported by
    MFA_PLAN_CHECK as MFA_ERR_DEVICE_CHECK, and the next clean call succeeds again."""
    case = inputs.small("noalloc_badblk", 2, [100, 200], seed=35)
    q, k, v, ks, vs, table, lens = _device(case)
    dec = mfa.Decoder(2, case.max_pages, case.num_blocks, host_seq_lens=case.seq_lens.tolist(),
                      flags=mfa.MFA_PLAN_CHECK)
    out = torch.empty((2, 64, 256), dtype=torch.bfloat16, device="cuda")
    bad = table.clone()
    bad[1, 2] = case.num_blocks + 7
    with pytest.raises(mfa.MfaError) as e:
        mfa.mfa_decode_run_static_workspace(dec.plan, dec.problem, q, k, v, ks, vs, bad, lens, out, None)
    assert e.value.status == mfa.MFA_ERR_DEVICE_CHECK
    mfa.mfa_decode_run_static_workspace(dec.plan, dec.problem, q, k, v, ks, vs, table, lens, out, None)
    torch.cuda.synchronize()
