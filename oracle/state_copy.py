"""State-pool gather/scatter as plain indexed copies (oracle).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Follows the numerical contract of the vllm-ascend article on the KDA prefill
state copy (section "数值契约", numerical contract):

Gather
  * a row whose index is out of range or negative, or whose flag is false,
    comes out as all zeros; without flags every valid row is gathered;
  * duplicate indices are legal (the same cache row is read again);
  * every packed row is written, invalid rows with zeros.
Scatter
  * invalid indices are skipped; valid targets are unique (a caller
    precondition, not checked);
  * flags describe only the initial state and never suppress a final write;
  * the packed state is first converted to the cache dtype.
Memory
  * only the payload of a row is copied: the gap between the payload and the
    next row (``row_stride - payload``) is neither read into the output nor
    overwritten; addresses are element offsets computed in 64 bits.
  * an empty selection copies nothing.

bf16 buffers are carried as their raw 16-bit patterns (``np.uint16``);
fp32 -> bf16 rounds to nearest, ties to even.
"""
from __future__ import annotations

import numpy as np


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the 16-bit patterns.

    Adding 0x7FFF plus the lowest kept bit to the 32-bit pattern and dropping
    the low half rounds to nearest with ties to even; NaNs stay quiet NaNs."""
    u = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32).astype(np.uint64)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r = np.where(nan, ((u >> 16) | 0x40).astype(np.uint16), r)
    return r


def bf16_bits_to_f32(b) -> np.ndarray:
    """Exact widening of bf16 patterns to fp32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rows(buf: np.ndarray, num_rows: int, row_stride: int, payload: int) -> np.ndarray:
    """[num_rows, payload] view of the payloads inside a flat element buffer."""
    return np.lib.stride_tricks.as_strided(
        buf, shape=(num_rows, payload), strides=(row_stride * buf.itemsize, buf.itemsize),
        writeable=buf.flags.writeable)


def _valid(idx, flags, num_rows):
    idx = np.asarray(idx, dtype=np.int64)
    ok = (idx >= 0) & (idx < num_rows)
    if flags is not None:
        ok &= np.asarray(flags, dtype=bool)
    return idx, ok


def state_gather(cache: np.ndarray, num_rows: int, row_stride: int, payload: int, idx,
                 flags=None) -> np.ndarray:
    """packed[i] = cache_row[idx[i]] if idx[i] valid (and flags[i]) else 0."""
    rows = _rows(cache, num_rows, row_stride, payload)
    idx, ok = _valid(idx, flags, num_rows)
    packed = np.zeros((len(idx), payload), dtype=cache.dtype)
    for i in range(len(idx)):
        if ok[i]:
            packed[i] = rows[idx[i]]
    return packed


def state_scatter(cache: np.ndarray, num_rows: int, row_stride: int, payload: int, idx,
                  packed: np.ndarray) -> np.ndarray:
    """Returns a copy of ``cache`` with cache_row[idx[i]] = cast(packed[i]) for
    every in-range idx[i].  ``packed`` fp32 into a bf16 (uint16) cache is
    rounded to nearest even; bf16 into fp32 widens exactly."""
    out = cache.copy()
    rows = _rows(out, num_rows, row_stride, payload)
    idx, ok = _valid(idx, None, num_rows)
    packed = np.asarray(packed).reshape(len(idx), payload)
    if out.dtype == packed.dtype:
        conv = packed
    elif out.dtype == np.uint16 and packed.dtype == np.float32:
        conv = f32_to_bf16_bits(packed)
    elif out.dtype == np.float32 and packed.dtype == np.uint16:
        conv = bf16_bits_to_f32(packed)
    else:
        raise TypeError("unsupported dtype pair")
    for i in range(len(idx)):
        if ok[i]:
            rows[idx[i]] = conv[i]
    return out
