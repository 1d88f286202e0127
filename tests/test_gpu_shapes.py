"""Parity of the comparison attention shapes (through the C ABI) with the fp64 CPU oracle.

The Step-3 page sets MFA against grouped-query attention and a latent shared by keys and
values (section 5 "Model-System Co-design", "Attention Design"; section 7, attention
ablation).  The same decode kernel family runs both:
  - grouped-query: 64 query heads of width 128 over 4 key/value heads (cache rows of 4 x 128);
  - shared latent: 128 query heads of width 512 over one 512-wide latent that is both the
    key and the value (no V pool).
Limits as for the bf16 MFA path: max-abs <= 1e-2 and relative-L2 <= 5e-3 on the fp32
output (half a bf16 ulp more for the bf16 output), lse within 2e-3; indexing exact
(NaN-poisoned unused slots and pages never reach the output).
"""
import numpy as np
import pytest
import torch

import decode_attention_02_gb300 as mfa
import oracle
from decode_attention_02_gb300 import inputs
from test_gpu_parity import BF16_MAX_ABS, BF16_REL_L2, check_parity, gpu_decode

pytestmark = pytest.mark.gpu

GQA = dict(head_dim=128, num_kv_heads=4)
MLA = dict(num_q_heads=128, head_dim=512, kv_shared=True)


@pytest.mark.parametrize("shape", ["gqa", "mla"])
@pytest.mark.parametrize("force_ctas", [0, 1, 3, 16, 64])
def test_ragged_lengths_any_split(shape, force_ctas):
    lens = [1, 63, 64, 65, 127, 128, 129, 200, 0, 517, 1000, 300]
    case = inputs.small(f"{shape}_r", len(lens), lens, seed=60, extra_blocks=3, **(GQA if shape == "gqa" else MLA))
    out, lse, _ = gpu_decode(case, force_ctas=force_ctas)
    check_parity(case, out, lse)


@pytest.mark.parametrize("shape", ["gqa", "mla"])
def test_bf16_output_is_rne_of_fp32_output(shape):
    case = inputs.small(f"{shape}_o", 4, [3000, 1, 700, 1500], seed=61, **(GQA if shape == "gqa" else MLA))
    o32, l32, _ = gpu_decode(case, force_ctas=5)
    o16, l16, _ = gpu_decode(case, force_ctas=5, out_dtype=mfa.MFA_OUT_BF16)
    assert torch.equal(o16.view(torch.int16), o32.to(torch.bfloat16).view(torch.int16))
    ref = oracle.decode(case)
    check_parity(case, o32, l32, ref=ref)
    check_parity(case, o16, l16, ref=ref)


def test_grouped_heads_use_only_their_key_value_head():
    """Poisoning key/value head 1's columns (NaN) leaves the 48 query heads of heads 0, 2, 3
    finite and equal to the oracle's; heads 16..31 go non-finite."""
    case = inputs.small("gqa_iso", 3, [100, 300, 64], seed=62, **GQA)
    ref_o, ref_l = oracle.decode(case)
    case.k_cache.view(torch.int16)[:, :, 128:256] = 0x7FC0
    out, lse, _ = gpu_decode(case, flags=0)
    got = out.double().cpu().numpy()
    keep = np.r_[0:16, 32:64]
    assert np.all(np.isfinite(got[:, keep]))
    assert np.abs(got[:, keep] - ref_o[:, keep]).max() <= BF16_MAX_ABS
    assert not np.isfinite(got[:, 16:32]).any()


def test_shared_latent_ignores_the_v_pointer():
    """With a shared latent the values are the key rows: the V pointer passed is not read."""
    case = inputs.small("mla_v", 3, [100, 300, 64], seed=63, **MLA)
    t = dict(q=case.q.cuda(), k=case.k_cache.cuda(), tb=case.block_table.cuda(), l=case.seq_lens.cuda())
    dec = mfa.Decoder(3, case.max_pages, case.num_blocks, host_seq_lens=case.seq_lens.tolist(),
                      flags=mfa.MFA_PLAN_CHECK, out_dtype=mfa.MFA_OUT_FP32, shape=mfa.SHAPE_MLA)
    out, lse = dec(t["q"], t["k"], None, t["tb"], t["l"])
    torch.cuda.synchronize()
    check_parity(case, out, lse)


def test_empty_sequences_give_zero_and_minus_inf():
    for kw in (GQA, MLA):
        case = inputs.small("shape_e", 4, [0, 70, 0, 1], seed=64, **kw)
        out, lse, _ = gpu_decode(case, force_ctas=2)
        check_parity(case, out, lse)
        assert float(out[0].abs().max()) == 0.0 and torch.isneginf(lse[0]).all()


@pytest.mark.parametrize("name", ["gqa_b32_l4096_bf16", "mla_b32_l4096_bf16"])
def test_full_size_workload(name):
    """The 4K comparison workloads in the bench's launch configuration, checked against the
    oracle on 8 of the 32 sequences (the oracle computes them one by one)."""
    case = inputs.generate(inputs.WORKLOADS[name])
    out, lse, dec = gpu_decode(case, flags=mfa.MFA_PLAN_CHECK | mfa.MFA_PLAN_EARLY_METADATA)
    units = 2 if case.workload.kv_shared else 1
    assert dec.plan.total_tiles == 32 * 32 * units
    sub = torch.tensor([0, 5, 11, 16, 21, 26, 30, 31])
    part = inputs.Case(workload=case.workload, q=case.q[sub].contiguous(), k_cache=case.k_cache,
                       v_cache=case.v_cache, k_scale=None, v_scale=None,
                       block_table=case.block_table[sub].contiguous(), seq_lens=case.seq_lens[sub].contiguous())
    ro, rl = oracle.decode(part)
    got = out.float().cpu().double().numpy()[sub.numpy()]
    err = np.abs(got - ro)
    rel = np.linalg.norm(got - ro) / np.linalg.norm(ro)
    assert err.max() <= BF16_MAX_ABS and rel <= BF16_REL_L2, (err.max(), rel)
    assert np.abs(lse.cpu().double().numpy()[sub.numpy()] - rl).max() <= 2e-3


@pytest.mark.parametrize("shape", ["gqa", "mla"])
def test_ctas_without_tiles(shape):
    """Cost ranges that hold no tile (here CTAs 3, 7 and 16 of 26 for grouped heads) do nothing."""
    lens = [1, 63, 64, 65, 127, 128, 129, 200, 0, 517, 1000, 300]
    case = inputs.small(f"{shape}_ec", len(lens), lens, seed=65, **(GQA if shape == "gqa" else MLA))
    out, lse, dec = gpu_decode(case, force_ctas=26)
    check_parity(case, out, lse)
