"""The algorithmic work the bench divides by (roofline `achieved`), pinned to
closed forms: causal prefill flops 4 D Hq sum(keys seen), with a prompt's
chunks partitioning the causal triangle; decode bytes = positions x KV heads
x bytes per position (bf16 K and V: 2 x 128 x 2; INT8 codes plus one fp32
scale each: 2 x (128 + 4))."""
import bench


def test_prefill_flops_of_a_1024_token_prompt():
    # every row i (1-based) sees i keys: 4 * 128 * 32 * 1024 * 1025 / 2
    assert bench.prefill_flops(1024, 1024, 32) == 8_598_323_200


def test_chunks_of_the_26926_token_prompt_sum_to_the_causal_triangle():
    N, chunk = 26926, 2048
    total = 0.0
    for lo in range(0, N, chunk):
        n = min(chunk, N - lo)
        total += bench.prefill_flops(n, lo + n, 32)
    assert total == 4.0 * 128 * 32 * N * (N + 1) // 2
    assert abs(total / 1e12 - 5.94) < 0.005


def test_a_chunk_sees_its_prefix_and_a_causal_square():
    # q rows after L - q cached positions: q (L - q) prefix keys + q (q + 1) / 2
    q, L = 300, 6000
    assert bench.prefill_flops(q, L, 8) == 4.0 * 128 * 8 * (q * (L - q) + q * (q + 1) // 2)


def test_decode_bytes_bf16_and_int8():
    assert bench.decode_bytes([1024], 8) == 4_194_304                 # 8 heads x 1k, bf16
    assert bench.decode_bytes([32768], 8, 264) == 69_206_016          # INT8, one sequence
    assert bench.decode_bytes([32768] * 8, 8, 264) == 553_648_128     # INT8, eight
