"""Work accounting (the roofline numerators) against hand counts."""
from qwen3_qk_norm_gb300 import accounting


def test_prefill_flops_counts_unmasked_pairs():
    # T = 3: pairs (0,0) (1,0) (1,1) (2,0) (2,1) (2,2) = 6, each 4 d flops per head
    assert accounting.prefill_flops(1, 3, 1, 128) == 6 * 4 * 128
    # the Qwen3-8B-shaped prefill: 4 * 128 * 32 * 4 * 4096 * 4097 / 2
    assert accounting.prefill_flops(4, 4096, 32) == 549890031616


def test_chunk_flops():
    # a chunk from position 0 is a prefill
    assert accounting.chunk_flops([0, 0], 100, 8) == accounting.prefill_flops(2, 100, 8)
    # one token after p cached tokens sees p + 1 keys
    assert accounting.chunk_flops([7], 1, 1, 128) == 8 * 4 * 128
    # chunks [0:2], [2:5], [5:6] add up to the prefill of 6 tokens
    parts = [accounting.chunk_flops([a], b - a, 4) for a, b in [(0, 2), (2, 5), (5, 6)]]
    assert sum(parts) == accounting.prefill_flops(1, 6, 4)


def test_decode_bytes_by_hand():
    # B = 1, Hq = 2, Hkv = 1, d = 128, start_pos 10: cache reads 10 rows of K and V,
    # inputs q (2 rows) + k_new + v_new + 2 gammas, writes 2 appended rows + 2 output rows
    row = 256
    want = 10 * 2 * row + (2 + 2) * row + 2 * row + 2 * row + 2 * row
    assert accounting.decode_bytes([10], 2, 1) == want


def test_gated_decode_bytes_count_query_and_gate_rows():
    from qwen3_qk_norm_gb300.accounting import gated_decode_bytes
    # one sequence at p = 10, Hq 2, Hkv 1, d 4 (2-byte elements):
    # cache 10 rows x (K + V) x 8 B = 160; q|gate 2 x 16 B + k_new, v_new 2 x 8 B + w's 16 B;
    # writes: appended K, V 16 B + out 2 x 8 B
    assert gated_decode_bytes([10], 2, 1, 4) == 160 + (32 + 16 + 16) + (16 + 16)


def test_chunk_flops_at_head_dim_256():
    """The gated chunk's work at d = 256: a chunk at position 0 is the gated
    prefill's work, and the bench's Qwen3-Next chunk (4 x 1024 tokens after
    3072 cached, 16 heads) is 4 * 256 * 16 * sum_b sum_t (3072 + t + 1)."""
    assert (accounting.chunk_flops([0, 0, 0], 50, 16, 256)
            == accounting.prefill_flops(3, 50, 16, 256))
    per_seq = sum(3072 + t + 1 for t in range(1024))
    assert accounting.chunk_flops([3072] * 4, 1024, 16, 256) == 4 * 256 * 16 * 4 * per_seq
    assert accounting.chunk_flops([3072] * 4, 1024, 16, 256) == 240551723008  # 4·256·16·4·(1024·3072 + 1024·1025/2)
