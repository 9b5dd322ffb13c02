"""The tiled MXFP4 layouts (1: rows, 2: gate/up pairs) and the UMMA layouts
(3: rows, 4: gate/up pairs) are byte permutations of the canonical packing,
laid out as the public header describes: checked on the host packer against a
direct numpy statement of that description, applied to the oracle's canonical
bytes."""
import numpy as np
import pytest
import torch

import oracle
import moe_decode_step_gb300 as M


def _tile_numpy(q, s, layout):
    """Canonical q [rows][k/2], s [rows][k/32] -> tiled byte arrays."""
    rows, kb = q.shape
    k = 2 * kb
    nblk = k // 32
    qt = np.full(rows * kb, 0xAB, np.uint8)
    st = np.full(rows * nblk, 0xAB, np.uint8)
    for row in range(rows):
        if layout == 2:
            n = rows // 2
            i, hi = (row, 0) if row < n else (row - n, 8)
            T, r = i // 8, i % 8 + hi
        else:
            T, r = row // 16, row % 16
        g, half = r % 8, r // 8
        for b in range(nblk):
            for u in range(4):   # lane (g, u) of block pair b // 2
                off = T * 8 * k + ((b // 2) * 32 + 4 * g + u) * 16 + (b % 2) * 8 + half * 4
                qt[off:off + 4] = q[row, 16 * b + 4 * u:16 * b + 4 * u + 4]
            st[T * (k // 2) + ((b // 4) * 8 + g) * 8 + (b % 4) * 2 + half] = s[row, b]
    return qt, st


def _umma_numpy(q, s, layout):
    """Canonical q [rows][k/2], s [rows][k/32] -> UMMA byte arrays."""
    rows, kb = q.shape
    k = 2 * kb
    nblk = k // 32
    qt = np.full(rows * kb, 0xAB, np.uint8)
    st = np.full(rows * nblk, 0xAB, np.uint8)
    for row in range(rows):
        if layout == 4:
            n = rows // 2
            i, hi = (row, 0) if row < n else (row - n, 64)
            T, m = i // 64, i % 64 + hi
        else:
            T, m = row // 128, row % 128
        for b in range(nblk):
            off = 64 * k * T + 2048 * b + 128 * (m // 8) + 16 * (m % 8)
            qt[off:off + 16] = q[row, 16 * b:16 * b + 16]
            st[4 * k * T + 512 * (b // 4) + 16 * (m % 32) + 4 * (m // 32) + b % 4] = s[row, b]
    return qt, st


@pytest.mark.parametrize("layout,rows,k", [(1, 32, 256), (2, 32, 256), (1, 16, 384),
                                           (2, 48, 128), (3, 128, 256), (4, 128, 384),
                                           (3, 256, 128), (4, 256, 128)])
def test_host_tiled_pack_is_the_documented_permutation(layout, rows, k):
    w = np.random.default_rng(rows * k + layout).standard_normal((rows, k)).astype(np.float32)
    qc, sc = oracle.mxfp4_pack(w)
    q, s = M.mxfp4_pack(torch.from_numpy(w), layout=layout)
    qt, st = (_umma_numpy if layout >= 3 else _tile_numpy)(qc, sc, layout)
    assert np.array_equal(q.numpy().ravel(), qt)
    assert np.array_equal(s.numpy().ravel(), st)


def test_tiled_layout_shape_rules():
    assert M.mxfp4_packed_bytes(16, 128, 1)[0] == 16 * 64
    assert M.mxfp4_packed_bytes(16, 96, 1)[0] == 0      # k % 128
    assert M.mxfp4_packed_bytes(24, 128, 2)[0] == 0     # whole tiles of 16 mma rows
    assert M.mxfp4_packed_bytes(24, 96, 0)[0] == 24 * 48
    assert M.mxfp4_packed_bytes(16, 128, 3)[0] == 0      # whole tiles of 128 mma rows
    assert M.mxfp4_packed_bytes(128, 128, 3)[0] == 128 * 64
    assert M.mxfp4_packed_bytes(128, 96, 4)[0] == 0
    assert M.mxfp4_packed_bytes(16, 128, 5)[0] == 0
    with pytest.raises(M.MoEError):
        M.mxfp4_pack(torch.zeros(24, 128), layout=1)


@pytest.mark.parametrize("layout", [1, 2, 3, 4])
def test_repack_round_trips_and_matches_the_tiled_packer(layout):
    w = np.random.default_rng(40 + layout).standard_normal((128, 256)).astype(np.float32)
    qc, sc = M.mxfp4_pack(torch.from_numpy(w), layout=0)
    qt, st = M.mxfp4_pack(torch.from_numpy(w), layout=layout)
    q1, s1 = M.mxfp4_repack(qc, sc, 0, layout)
    assert torch.equal(q1, qt) and torch.equal(s1, st)
    q2, s2 = M.mxfp4_repack(qt, st, layout, 0)
    assert torch.equal(q2, qc) and torch.equal(s2, sc)
    for other in (1, 2, 3, 4):
        if other != layout:
            q3, s3 = M.mxfp4_repack(*M.mxfp4_repack(qt, st, layout, other), other, layout)
            assert torch.equal(q3, qt) and torch.equal(s3, st)
