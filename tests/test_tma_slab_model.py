"""Model check of the weight-slab loads of the dX-chain products (no GPU).

BWD2T and BWD1T read their weight operand N-major, as four 64-column slabs of [64 K rows]
x [64 columns] placed one after the other in shared memory, each row a 128-byte line under
the 128-byte swizzle (16-byte chunk c of line L stored at chunk c ^ (L % 8)). They used to
issue four 3-D tensor copies (box {64, 64, 1} at column offsets 0, 64, 128, 192) and now
issue one 4-D copy of the view {64, rows, cols / 64, n} with strides {a row, 128 bytes,
a matrix} and box {64, 64, 4, 1}. The functions below emulate a tiled tensor copy (box
elements in dimension order, out-of-range elements zero, swizzle on the destination lines)
and check that both forms write the same bytes, including a last N tile that runs past the
columns.
"""
import numpy as np
import pytest


def tiled_copy(mem, dims, strides, box, coords):
    """Elements of one box, innermost dimension fastest, as a flat list (0 out of range).
    mem: flat element array; dims / strides / coords in elements, dimension 0 innermost."""
    out = []

    def rec(level, offset, inb):
        if level < 0:
            out.append(mem[offset] if inb else 0)
            return
        for i in range(box[level]):
            c = coords[level] + i
            ok = inb and 0 <= c < dims[level]
            rec(level - 1, offset + (c * strides[level] if ok else 0), ok)

    rec(len(dims) - 1, 0, True)
    return np.array(out, dtype=mem.dtype)


def swizzle128(elems_bf16):
    """Place a run of 128-byte lines (64 bf16 each) under the 128-byte swizzle."""
    lines = elems_bf16.reshape(-1, 8, 8)          # [line][16-byte chunk of 8 bf16]
    out = np.empty_like(lines)
    for L in range(lines.shape[0]):
        for c in range(8):
            out[L, c ^ (L % 8)] = lines[L, c]
    return out.reshape(-1)


@pytest.mark.parametrize("rows,cols,n,k0,n0,e", [(128, 512, 2, 64, 256, 1), (192, 320, 3, 128, 256, 2),
                                                 (64, 256, 1, 0, 0, 0)])
def test_one_4d_copy_lands_the_four_slabs(rows, cols, n, k0, n0, e):
    rng = np.random.default_rng(rows + cols)
    mem = rng.integers(1, 2**15, size=n * rows * cols).astype(np.int32)   # [n][rows][cols]
    # four 3-D copies: view {cols, rows, n}, box {64, 64, 1}, column offsets n0 + 64 i
    four = np.concatenate([
        tiled_copy(mem, [cols, rows, n], [1, cols, rows * cols], [64, 64, 1], [n0 + 64 * i, k0, e])
        for i in range(4)])
    # one 4-D copy: view {64, rows, cols / 64, n}, strides {1, cols, 64, rows * cols}
    one = tiled_copy(mem, [64, rows, cols // 64, n], [1, cols, 64, rows * cols], [64, 64, 4, 1],
                     [0, k0, n0 // 64, e])
    assert one.size == four.size == 4 * 64 * 64
    assert np.array_equal(swizzle128(one), swizzle128(four))
    # the slabs past the last column are zero in both (the tile's ragged N end)
    past = max(0, (n0 + 256 - cols) // 64)
    if past:
        assert not one[(4 - past) * 4096:].any()
