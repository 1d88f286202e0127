"""The benchmark's algorithmic-work accounting, written out by hand for small cases.

Per cached token and sequence, decode attention with H heads of width d moves 2*d K/V values
(2 bytes each in bf16, 1 byte plus two fp32 scales in e4m3) and does 4*H*d FLOPs (q.K^T and
P.V).  With T new query tokens per sequence, query token i of a sequence of L tokens sees
L - T + 1 + i of them; the cache is still read once, while q, out and lse are per query token.
"""
import bench

H, D = 64, 256


def test_single_token_bytes_and_flops():
    lens = [1, 64, 65, 0]
    a = bench.algorithmic_bytes(lens, "bf16")
    assert a["kv"] == 130 * 2 * D * 2
    pages = 1 + 1 + 2 + 0
    assert a["total"] == a["kv"] + 4 * (H * D * 2) * 2 + pages * 4 + 4 * 4 + 4 * H * 4
    e = bench.algorithmic_bytes(lens, "fp8_e4m3")
    assert e["kv"] == 130 * (2 * D + 2 * 4)
    assert bench.algorithmic_flops(lens) == 130 * 4 * H * D


def test_multi_token_counts_pairs_and_reads_the_cache_once():
    lens, T = [10, 1, 0], 2
    # query tokens see 9 and 10 tokens (L = 10), 0 and 1 (L = 1), nothing (L = 0)
    assert bench.algorithmic_flops(lens, T=T) == (9 + 10 + 0 + 1) * 4 * H * D
    a = bench.algorithmic_bytes(lens, "bf16", T=T)
    one = bench.algorithmic_bytes(lens, "bf16")
    assert a["kv"] == one["kv"]
    assert a["total"] - one["total"] == 3 * (T - 1) * (H * D * 2 * 2 + H * 4)


def test_append_bytes():
    # per sequence: two bf16 rows in, position and page id, two rows out
    assert bench.append_bytes(3, "bf16") == 3 * (2 * 2 * D + 4 + 4 + 2 * 2 * D)
    assert bench.append_bytes(3, "fp8_e4m3") == 3 * (2 * 2 * D + 4 + 4 + 2 * (D + 4))
    # T new tokens per sequence: one position per sequence, rows and page ids per token
    assert bench.append_bytes(3, "bf16", T=2) == 3 * (4 + 2 * (2 * 2 * D + 4 + 2 * 2 * D))
