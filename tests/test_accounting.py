"""The benchmark's algorithmic byte counts, the numerator of every roofline
figure it reports, checked against the per-token sizes of the cache layout
(include/qs.h): per (token, head) a draft reads the upper key and value
nibbles (64 B + 64 B) and its share of the group's scales and zero-points
(1 KB per 128 tokens = 8 B); verify adds the two lower planes (128 B); the
two-bit draft reads half of each upper plane (32 B + 32 B). A buffer token is
fp16 K and V (2 x 256 B); a query row and an output row are 256 B each."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

G, D = 128, 128
ROW = D * 2                     # one fp16 row of 128 channels
META_PER_TOKEN = 4 * D * 2 // G  # four fp16 vectors of 128 per group


@pytest.mark.parametrize("ng, fill, n_q, BH", [(0, 1, 1, 1), (255, 129, 1, 32), (1023, 133, 5, 32),
                                               (7, 64, 8, 3)])
def test_attention_bytes_follow_the_layout(ng, fill, n_q, BH):
    tokens = ng * G
    draft = BH * (tokens * (D // 2 + D // 2 + META_PER_TOKEN) + fill * 2 * ROW + n_q * 2 * ROW)
    verify = BH * (tokens * (4 * (D // 2) + META_PER_TOKEN) + fill * 2 * ROW + n_q * 2 * ROW)
    two_bit = BH * (tokens * (D // 4 + D // 4 + META_PER_TOKEN) + fill * 2 * ROW + n_q * 2 * ROW)
    assert bench.attn_bytes(ng, fill, n_q, True, BH) == draft
    assert bench.attn_bytes(ng, fill, n_q, False, BH) == verify
    assert bench.attn_bytes(ng, fill, n_q, True, BH, upper_bits=2) == two_bit
    # verify re-reads nothing the two-bit layout saves: its bytes do not depend on it
    assert bench.attn_bytes(ng, fill, n_q, False, BH, upper_bits=2) == verify


def test_per_token_head_figures():
    """136 B (draft), 264 B (verify), 72 B (two-bit draft) per token-head."""
    per = lambda **k: (bench.attn_bytes(2, 0, 0, BH=1, **k) - bench.attn_bytes(1, 0, 0, BH=1, **k)) / G
    assert per(mode_draft=True) == 136
    assert per(mode_draft=False) == 264
    assert per(mode_draft=True, upper_bits=2) == 72


def test_grouped_query_heads_add_only_query_and_output_rows():
    base = bench.attn_bytes(255, 129, 5, False, 8)
    assert bench.attn_bytes(255, 129, 5, False, 8, group=4) - base == 8 * 3 * 5 * 2 * ROW


def test_flush_and_append_bytes():
    # a flush reads the oldest half's K and V rows and writes four 8 KB planes
    # plus 1 KB of scales and zero-points
    assert bench.FLUSH_BYTES_PER_HEAD == 2 * G * ROW + 4 * G * (D // 2) + G * META_PER_TOKEN
    # an append reads the new tokens' K and V rows and writes them into the ring
    assert bench.append_bytes(5, 32) == 32 * 5 * (2 * ROW + 2 * ROW)


@pytest.mark.parametrize("L", [0, 1, 256, 257, 384, 385, 32768])
def test_prefill_bytes(L):
    """Read the prompt's K and V; write the groups (all four planes plus
    metadata) and the buffer tokens; the split is ceil((L - 2G) / G) groups."""
    ng = max(0, -(-(L - 2 * G) // G))
    rest = L - ng * G
    assert 0 <= rest <= 2 * G
    want = L * 2 * ROW + ng * G * (4 * (D // 2) + META_PER_TOKEN) + rest * 2 * ROW
    assert bench.prefill_bytes(L, 1) == want
    assert bench.prefill_bytes(L, 32) == 32 * want


def test_32k_round_bytes():
    """The benchmark step on the 32k workload (32 heads, a 32,768-token
    context whose last 2G tokens fill the buffer): the flush retires one half
    (255 groups, 128 buffered tokens after it), then four drafts over 129..132
    buffered tokens, four appended tokens rolled back, five appended, one
    5-query verify over 133."""
    from hierarchical_quantized_kv_gb300 import synthetic
    w = synthetic.CONFIGS["32k"]()
    H, L = 32, 32768
    assert (w.H, w.context[0], w.fill[0]) == (H, L, 2 * G)
    groups = (L - 2 * G) // G + 1
    assert groups == 255
    tok = groups * G
    flush = H * (2 * G * ROW + G * (4 * (D // 2) + META_PER_TOKEN))
    drafts = sum(H * (tok * 136 + (G + 1 + i) * 2 * ROW + 2 * ROW) for i in range(4))
    verify = H * (tok * 264 + (G + 5) * 2 * ROW + 5 * 2 * ROW)
    appends = H * 9 * 4 * ROW
    total = flush + drafts + verify + appends
    assert total == 858_292_224  # the bench line's bytes_per_step
    ng1, f1 = w.n_groups[0] + 1, w.fill[0] - w.G
    got = (bench.FLUSH_BYTES_PER_HEAD * H
           + sum(bench.attn_bytes(ng1, f1 + i + 1, 1, True, H) for i in range(bench.GAMMA))
           + bench.attn_bytes(ng1, f1 + bench.GAMMA + 1, bench.GAMMA + 1, False, H)
           + bench.append_bytes(bench.GAMMA, H) + bench.append_bytes(bench.GAMMA + 1, H))
    assert got == total


def _seq_draft(ng, fill, H):
    return H * (ng * G * 136 + fill * 2 * ROW + 2 * ROW)


def _seq_verify(ng, fill, H, n_q=5):
    return H * (ng * G * 264 + fill * 2 * ROW + n_q * 2 * ROW)


def test_round_plan_counts_each_sequence_from_its_own_counters():
    """A batch whose sequences differ: only those whose buffer cannot take
    the five target tokens (fill + 5 > 2G) flush, and each sequence's drafts
    and verify read its own groups and buffered tokens."""
    H = 2
    ng0, f0 = [10, 3, 0, 7], [256, 40, 251, 252]
    p = bench.round_plan(ng0, f0, H)
    assert list(p["mask"]) == [1, 0, 0, 1]
    assert list(p["ng1"]) == [11, 3, 0, 8] and list(p["f1"]) == [128, 40, 251, 124]
    assert p["bytes"]["flush"] == 2 * H * (2 * G * ROW + G * (4 * (D // 2) + META_PER_TOKEN))
    for i in range(4):
        assert p["bytes"]["draft"][i] == sum(_seq_draft(n, f + i + 1, H)
                                             for n, f in zip(p["ng1"], p["f1"]))
    assert p["bytes"]["verify"] == sum(_seq_verify(n, f + 5, H) for n, f in zip(p["ng1"], p["f1"]))
    assert p["bytes"]["append"] == 4 * H * 9 * (2 * ROW + 2 * ROW)  # 4 sequences, 9 tokens
    assert p["step"] == (p["bytes"]["flush"] + sum(p["bytes"]["draft"]) + p["bytes"]["verify"]
                         + p["bytes"]["append"])


def test_ragged_and_batched_rounds():
    """The ragged workload (16 sequences, contexts 4k..64k, fill 1..256) and
    the batched one (8 x 32k): bytes summed over sequences from their own
    counters, flushes only where due."""
    from hierarchical_quantized_kv_gb300 import synthetic
    for w in (synthetic.ragged(), synthetic.batched_32k()):
        p = bench.round_plan(w.n_groups, w.fill, w.H)
        due = [f + 5 > 2 * G for f in w.fill]
        assert list(p["mask"]) == [int(x) for x in due]
        ng1 = [n + d for n, d in zip(w.n_groups, due)]
        f1 = [f - G * d for f, d in zip(w.fill, due)]
        want_draft = sum(_seq_draft(n, f + 1, w.H) for n, f in zip(ng1, f1))
        assert p["bytes"]["draft"][0] == want_draft
        assert p["bytes"]["verify"] == sum(_seq_verify(n, f + 5, w.H) for n, f in zip(ng1, f1))
        assert p["bytes"]["flush"] == sum(due) * w.H * bench.FLUSH_BYTES_PER_HEAD
    w = synthetic.ragged()
    assert 0 < sum(f + 5 > 2 * G for f in w.fill) < w.B   # some flush, some do not
    # the 32k round seen through the plan: the bench line's 858,292,224 bytes
    w = synthetic.llama_32k()
    assert bench.round_plan(w.n_groups, w.fill, w.H)["step"] == 858_292_224


def test_oracle_sample_bytes():
    """The CPU baseline's sample: sequence 0's counters on the sampled heads."""
    from hierarchical_quantized_kv_gb300 import synthetic
    w = synthetic.llama_32k()
    assert bench.sample_step_bytes(w, 32) == 858_292_224
    assert bench.sample_step_bytes(w, 16) * 2 == 858_292_224
