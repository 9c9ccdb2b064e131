"""Alignment of every bulk async copy the kernels issue, for every supported
row count and head size: a copy must start and end on a 16-byte boundary
(shared and global side).  The layout formulas mirror csrc/gdn_spec.cu's
`Stage`, `gram_floats` and `work_floats`; `gdn_work_bytes` is checked against
them through the library."""
from __future__ import annotations

import itertools

import pytest


def gram_floats(R):
    return (2 * R * R + 3) & ~3


def dvs(dk):
    return 16 if dk == 16 else 32


@pytest.mark.parametrize("dk", [16, 32, 64, 128])
def test_rows_kernel_stage_and_copies_are_16_byte_aligned(dk):
    D = dvs(dk)
    for R in range(1, 17):
        rfl = R * 2 * dk + R * D + R * 4 + gram_floats(R)
        for s in (0, 1):
            qk = D * dk + s * rfl
            v = qk + R * 2 * dk
            sc = v + R * D
            gh = sc + R * 4
            for off in (qk, v, sc, gh):
                assert off % 4 == 0, (dk, R, s, off)
        for rows in range(1, R + 1):
            for nbytes in (D * dk * 4, rows * 2 * dk * 4, rows * D * 4, rows * 16, gram_floats(R) * 4):
                assert nbytes % 16 == 0, (dk, R, rows, nbytes)


@pytest.mark.parametrize("dk,B,R,Hq,G", list(itertools.product([16, 128], [1, 3], [1, 3, 9, 16], [1, 2], [1, 4])))
def test_work_regions_are_16_byte_aligned(cuda_lib, dk, B, R, Hq, G):
    Hv, dv = Hq * G, dvs(dk) * 2
    slices = dv // dvs(dk)
    qk = B * R * Hq * 2 * dk
    v = B * R * Hv * dv
    sc = B * R * Hv * 4
    total = qk + v + sc + B * Hq * gram_floats(R)
    for off in (qk, qk + v, qk + v + sc, total):
        assert off % 4 == 0
    # the per-item runs inside each region
    for b in range(B):
        for hq in range(Hq):
            assert ((b * Hq + hq) * R * 2 * dk) % 4 == 0
            assert ((b * Hq + hq) * gram_floats(R)) % 4 == 0
        for hs in range(Hv * slices):
            assert ((b * Hv * slices + hs) * R * dvs(dk)) % 4 == 0
        for h in range(Hv):
            assert ((b * Hv + h) * R * 4) % 4 == 0
    a = cuda_lib.GdnArgs(B=B, R=R, H_qk=Hq, H_v=Hv, d_k=dk, d_v=dv, W=4, pool_slots=1,
                         in_dtype=cuda_lib.BF16, scale=1.0, l2_eps=1e-6, flags=0)
    assert cuda_lib.work_bytes(a) == 4 * total
