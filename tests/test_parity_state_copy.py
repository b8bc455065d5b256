"""GPU gather/scatter against the oracle: bit-exact, through the C ABI.

Cases follow the behaviours the state-copy contract lists: gap between
payload and row stride, a storage offset, invalid and duplicate indices,
false flags, int32 and int64 indices, dtype conversion on scatter, an empty
selection, and rows more than 4 GiB apart."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def _bits(t):
    """Raw element patterns as numpy (uint16 for bf16, float32 view otherwise)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _pool(rows, payload_shape, gap, dtype, offset=0, seed=0):
    """A pool whose rows are `gap` elements longer than the payload, placed
    `offset` elements into its storage; the gap holds a canary."""
    g = torch.Generator().manual_seed(seed)
    payload = int(np.prod(payload_shape))
    stride = payload + gap
    flat = torch.full((offset + rows * stride,), 7.25, dtype=torch.float32)
    flat[offset:].view(rows, stride)[:, :payload] = torch.randn(rows, payload, generator=g)
    flat = flat.to(dtype).cuda()
    view = flat[offset:].as_strided((rows, *payload_shape),
                                    (stride, *torch.empty(payload_shape).stride()))
    return flat, view, stride, payload


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("idx_dtype", [torch.int32, torch.int64])
@pytest.mark.parametrize("gap,offset", [(0, 0), (8, 16), (3, 5)])
def test_gather_bit_exact(cuda_lib, dtype, idx_dtype, gap, offset):
    rows, shape = 9, (2, 8, 16)
    flat, pool, stride, payload = _pool(rows, shape, gap, dtype, offset)
    idx = torch.tensor([3, -1, 8, 3, 9, 0, 100, 5], dtype=idx_dtype, device="cuda")
    flags = torch.tensor([1, 1, 1, 0, 1, 1, 1, 1], dtype=torch.bool, device="cuda")
    before = _bits(flat)
    packed = cuda_lib.kda_state_gather(pool, idx, flags)
    ref = oracle.state_gather(_bits(flat)[offset:], rows, stride, payload, idx.cpu().numpy(),
                              flags.cpu().numpy())
    np.testing.assert_array_equal(_bits(packed).reshape(len(idx), payload), ref)
    np.testing.assert_array_equal(_bits(flat), before)  # the pool is only read
    packed2 = cuda_lib.kda_state_gather(pool, idx)       # no flags
    ref2 = oracle.state_gather(_bits(flat)[offset:], rows, stride, payload, idx.cpu().numpy())
    np.testing.assert_array_equal(_bits(packed2).reshape(len(idx), payload), ref2)


@pytest.mark.parametrize("cache_dtype,packed_dtype", [(torch.float32, torch.float32),
                                                      (torch.bfloat16, torch.float32),
                                                      (torch.float32, torch.bfloat16),
                                                      (torch.bfloat16, torch.bfloat16)])
@pytest.mark.parametrize("gap,offset", [(0, 0), (8, 16), (3, 5)])
def test_scatter_bit_exact(cuda_lib, cache_dtype, packed_dtype, gap, offset):
    rows, shape = 7, (2, 8, 16)
    flat, pool, stride, payload = _pool(rows, shape, gap, cache_dtype, offset, seed=1)
    idx = torch.tensor([4, -1, 0, 7, 2], dtype=torch.int64, device="cuda")
    packed = (torch.randn(len(idx), *shape, generator=torch.Generator().manual_seed(2)) * 3
              ).to(packed_dtype).cuda()
    before = _bits(flat)
    cuda_lib.kda_state_scatter(pool, idx, packed)
    ref = oracle.state_scatter(before[offset:].copy(), rows, stride, payload, idx.cpu().numpy(),
                               _bits(packed).reshape(len(idx), payload))
    got = _bits(flat)
    np.testing.assert_array_equal(got[:offset], before[:offset])   # storage before the pool
    np.testing.assert_array_equal(got[offset:], ref)               # rows and gaps


def test_empty_selection_launches_nothing(cuda_lib):
    flat, pool, _, _ = _pool(3, (4, 8), 0, torch.float32)
    idx = torch.empty(0, dtype=torch.int32, device="cuda")
    packed = cuda_lib.kda_state_gather(pool, idx)
    assert packed.shape == (0, 4, 8)
    cuda_lib.kda_state_scatter(pool, idx, packed)


def test_rows_more_than_4_gib_apart(cuda_lib):
    """Row stride * element size > 2^32 with int32 indices."""
    payload = 64
    stride = (1 << 30) + 64          # fp32: 4 GiB + 256 B between rows
    flat = torch.zeros(stride + payload, dtype=torch.float32, device="cuda")
    pool = flat.as_strided((2, payload), (stride, 1))
    pool[1] = torch.arange(payload, dtype=torch.float32, device="cuda")
    idx = torch.tensor([1, 0, 1], dtype=torch.int32, device="cuda")
    packed = cuda_lib.kda_state_gather(pool, idx)
    torch.testing.assert_close(packed[0], pool[1], rtol=0, atol=0)
    torch.testing.assert_close(packed[1], pool[0], rtol=0, atol=0)
    new = torch.full((1, payload), -3.0, device="cuda")
    cuda_lib.kda_state_scatter(pool, torch.tensor([1], dtype=torch.int32, device="cuda"), new)
    torch.testing.assert_close(pool[1], new[0], rtol=0, atol=0)
    assert float(flat[payload:stride].abs().max()) == 0.0   # the gap is untouched
    del flat, pool
    torch.cuda.empty_cache()
