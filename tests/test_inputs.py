"""The seeded generator follows the stated recipe (shapes, lengths, layouts, FP8 storage)."""
import numpy as np
import torch

from decode_attention_02_gb300 import inputs


def test_ragged_lengths_and_spikes():
    w = inputs.WORKLOADS["ragged_b128_l1024_8192_bf16"]
    lens = np.random.default_rng(w.seed).integers(1024, 8193, size=w.batch)
    assert lens.min() >= 1024 and lens.max() <= 8192
    # the spike rate: Bernoulli(0.01) per scalar, checked on a small pool
    small = inputs.Workload("s", batch=2, lens=(640, 640), seed=3, k_spike_frac=0.01, poison=False)
    c = inputs.generate(small)
    big = (c.k_cache.float().abs() > 6.0).float().mean().item()
    assert 0.004 < big < 0.012


def test_shuffled_table_is_a_bijection_onto_used_blocks():
    c = inputs.small("t", 4, [1, 64, 65, 300], extra_blocks=5)
    t = c.block_table.numpy()
    used = t[t >= 0]
    assert len(set(used.tolist())) == len(used) == 1 + 1 + 2 + 5
    assert used.max() < c.num_blocks
    # pages past each sequence's length are marked unused
    for b, L in enumerate(c.seq_lens.tolist()):
        n = (L + 63) // 64
        assert (t[b, :n] >= 0).all() and (t[b, n:] == -1).all()


def test_contiguous_layout_is_identity():
    c = inputs.generate(inputs.WORKLOADS["tiny_b1_l512_bf16"])
    assert c.block_table.tolist() == [list(range(8))]
    assert c.q.shape == (1, 64, 256) and c.q.dtype == torch.bfloat16


def test_fp8_storage_scales_are_absmax_over_448():
    c = inputs.small("f", 2, [64, 100], kv_dtype="fp8_e4m3", extra_blocks=0, seed=9)
    codes = c.k_cache.view(torch.float8_e4m3fn).to(torch.float64)
    t = c.block_table
    blk = int(t[0, 0])
    # every full row uses the top code magnitude 448 exactly once at least
    assert torch.all(codes[blk].abs().amax(dim=-1) == 448.0)
    assert torch.all(c.k_scale[blk] > 0)


def test_poison_marks_tails_and_unused_blocks():
    c = inputs.small("p", 1, [70], extra_blocks=2)
    t = c.block_table
    last = int(t[0, 1])
    assert torch.isnan(c.k_cache[last, 6:].float()).all()
    assert torch.isfinite(c.k_cache[last, :6].float()).all()
    unused = sorted(set(range(c.num_blocks)) - set(t[t >= 0].tolist()))
    assert len(unused) == 2 and torch.isnan(c.v_cache[unused].float()).all()


def test_generation_is_deterministic():
    a = inputs.small("d", 2, [33, 77], seed=5)
    b = inputs.small("d", 2, [33, 77], seed=5)
    assert torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16))
    assert torch.equal(a.block_table, b.block_table)
