"""The workspace-free decode entry point gives the same results as the regular one.

mfa_decode_run_static_workspace serves callers that cannot allocate device
memory themselves (for instance a plugin whose host application owns every
device allocation, or a latency-critical path that must not pay cudaMalloc's
implicit synchronisation): it uses a fixed scratch array that lives inside the
library.  These checks call it through the C ABI twice in a row, on two
different batches, and compare each result with mfa_decode_run's under the
limits the parity tests use.  The file is named so that pytest collects it
last.
"""
import numpy as np
import pytest
import torch

import decode_attention_02_gb300 as mfa
from decode_attention_02_gb300 import inputs

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2, LSE_ABS = 1e-2, 5e-3, 2e-3


def _device(case):
    d = "cuda"
    return (case.q.to(d), case.k_cache.to(d), case.v_cache.to(d), case.block_table.to(d), case.seq_lens.to(d))


def _close(a, b):
    a = a.float().cpu().double().numpy()
    b = b.float().cpu().double().numpy()
    err = np.abs(a - b)
    allow = MAX_ABS + np.abs(b) * 2.0 ** -8          # both outputs are bf16
    rel = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
    return bool(np.all(err <= allow)) and rel <= REL_L2


def test_static_workspace_matches_regular_entry_point_on_two_calls_in_a_row():
    cases = [inputs.small("noalloc_a", 7, [4096, 1000, 64, 2500, 1, 3000, 0], seed=31, k_spike_frac=0.01),
             inputs.small("noalloc_b", 3, [129, 700, 8000], seed=32)]
    for case in cases:
        q, k, v, table, lens = _device(case)
        B = case.q.shape[0]
        # regular entry point, workspace from PyTorch
        dec = mfa.Decoder(B, case.max_pages, case.num_blocks, host_seq_lens=case.seq_lens.tolist())
        out_r, lse_r = dec(q, k, v, table, lens)
        # workspace-free entry point: same plan and problem, no workspace argument
        out_s = torch.full_like(out_r, float("nan"))
        lse_s = torch.full_like(lse_r, float("nan"))
        mfa.mfa_decode_run_static_workspace(dec.plan, dec.problem, q, k, v, None, None, table, lens, out_s, lse_s)
        torch.cuda.synchronize()
        assert dec.plan.workspace_bytes <= mfa.MFA_STATIC_WORKSPACE_BYTES
        assert torch.isfinite(out_s.float()).all()
        assert _close(out_s, out_r)
        fin = torch.isfinite(lse_r)
        assert torch.equal(fin, torch.isfinite(lse_s))
        assert (lse_s[fin] - lse_r[fin]).abs().max().item() <= LSE_ABS


def test_static_workspace_rejects_plans_that_do_not_fit():
    B = 400
    prob = mfa.make_problem(B, 1, 4)
    plan = mfa.mfa_decode_plan(prob, None, max_seq_len=64, num_sms=152)
    assert plan.workspace_bytes > mfa.MFA_STATIC_WORKSPACE_BYTES
    small = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(mfa.MfaError) as e:
        mfa.mfa_decode_run_static_workspace(plan, prob, small, small, small, None, None, small, small, small, None)
    assert e.value.status == mfa.MFA_ERR_WORKSPACE
