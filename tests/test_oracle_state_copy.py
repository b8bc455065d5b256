"""Pins of the gather/scatter oracle against hand-worked cases of the state
copy contract (vllm-ascend KDA prefill state copy article, section
"数值契约"), and of its fp32 -> bf16 rounding against torch's conversion."""
import numpy as np
import torch

from oracle import state_gather, state_scatter, f32_to_bf16_bits, bf16_bits_to_f32

# 3 rows, payload 2, row stride 3: the third element of each row is gap (99).
CACHE = np.array([1, 2, 99, 3, 4, 99, 5, 6, 99], dtype=np.float32)


def test_gather_invalid_rows_are_zero_and_duplicates_legal():
    idx = [2, -1, 0, 2, 7]
    flags = [True, True, False, True, True]
    packed = state_gather(CACHE, 3, 3, 2, idx, flags)
    np.testing.assert_array_equal(packed, [[5, 6], [0, 0], [0, 0], [5, 6], [0, 0]])


def test_gather_without_flags_reads_every_valid_row():
    packed = state_gather(CACHE, 3, 3, 2, [1, 1, 3])
    np.testing.assert_array_equal(packed, [[3, 4], [3, 4], [0, 0]])


def test_scatter_skips_invalid_ignores_gap():
    packed = np.array([[10, 11], [12, 13], [14, 15], [16, 17]], dtype=np.float32)
    out = state_scatter(CACHE, 3, 3, 2, [2, -1, 0, 5], packed)
    np.testing.assert_array_equal(out, [14, 15, 99, 3, 4, 99, 10, 11, 99])
    np.testing.assert_array_equal(CACHE, [1, 2, 99, 3, 4, 99, 5, 6, 99])  # input untouched


def test_empty_selection():
    assert state_gather(CACHE, 3, 3, 2, []).shape == (0, 2)
    np.testing.assert_array_equal(state_scatter(CACHE, 3, 3, 2, [], np.zeros((0, 2), np.float32)), CACHE)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-40, 38, 20000),
        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 3.3895314e38, np.inf, -np.inf,
                  1e-40, -0.0, 0.0], dtype=np.float32)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(f32_to_bf16_bits(x), ref)
    # ties go to even: 1 + 2^-8 -> 1.0 (0x3F80); 1 + 3*2^-8 -> 0x3F82
    assert f32_to_bf16_bits(np.float32(1.0 + 2 ** -8)) == 0x3F80
    assert f32_to_bf16_bits(np.float32(1.0 + 3 * 2 ** -8)) == 0x3F82
    assert np.isnan(bf16_bits_to_f32(f32_to_bf16_bits(np.float32(np.nan))))


def test_scatter_fp32_into_bf16_cache_rounds():
    cache = np.zeros(6, dtype=np.uint16)
    packed = np.array([[1.0 + 2 ** -8, 2.5, -7.0]], dtype=np.float32)
    out = state_scatter(cache, 2, 3, 3, [1], packed)
    np.testing.assert_array_equal(out[3:], f32_to_bf16_bits(packed[0]))
    np.testing.assert_array_equal(out[:3], 0)
    np.testing.assert_array_equal(bf16_bits_to_f32(out[3:]), [1.0, 2.5, -7.0])
