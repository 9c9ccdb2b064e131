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


# state rows per item: every d_k's two-warp (or one-warp) geometry, and the
# four-warp 64-row geometry at d_k = 128
GEOMETRIES = [(16, 16), (32, 32), (64, 32), (128, 32), (128, 64)]


@pytest.mark.parametrize("dk,D", GEOMETRIES)
def test_rows_kernel_stage_and_copies_are_16_byte_aligned(dk, D):
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
@pytest.mark.parametrize("wide", [False, True])
def test_work_regions_are_16_byte_aligned(cuda_lib, dk, B, R, Hq, G, wide):
    if wide and dk != 128:
        pytest.skip("the 64-row geometry is for d_k = 128")
    D = 64 if wide else dvs(dk)
    Hv, dv = Hq * G, D * 2
    slices = dv // D
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
            assert ((b * Hv * slices + hs) * R * D) % 4 == 0
        for h in range(Hv):
            assert ((b * Hv + h) * R * 4) % 4 == 0
    a = cuda_lib.GdnArgs(B=B, R=R, H_qk=Hq, H_v=Hv, d_k=dk, d_v=dv, W=4, pool_slots=1,
                         in_dtype=cuda_lib.BF16, scale=1.0, l2_eps=1e-6, flags=0)
    assert cuda_lib.work_bytes(a) == 4 * total


def round4(r):
    return (r + 3) & ~3


@pytest.mark.parametrize("dk", [16, 32, 64, 128])
def test_deferred_staging_and_carry_copies_are_16_byte_aligned(dk):
    """Deferred mode stages, after an item's rows, the pending rows' carry:
    [Rp][DVS] update vectors, [Rp][d_k] k^, [Rp4] decays; with one or two
    staging buffers every region and every copy is a multiple of 16 bytes."""
    D = dvs(dk)
    for R in range(1, 17):
        for Rp in range(0, 17):
            carry = Rp * D + Rp * dk + round4(Rp)
            rfl = R * 2 * dk + R * D + R * 4 + gram_floats(R) + carry
            for stages in (1, 2):
                for s in range(stages):
                    base = D * dk + s * rfl
                    cu = base + R * 2 * dk + R * D + R * 4 + gram_floats(R)
                    ck = cu + Rp * D
                    ca = ck + Rp * dk
                    for off in (cu, ck, ca, base + rfl):
                        assert off % 4 == 0, (dk, R, Rp, stages, off)
            for prev in range(1, Rp + 1):
                for nbytes in (prev * D * 4, prev * dk * 4, round4(prev) * 4):
                    assert nbytes % 16 == 0


@pytest.mark.parametrize("dk,B,R,Hq,G", list(itertools.product([16, 128], [1, 3], [1, 4, 9, 16], [1, 2], [1, 4])))
def test_carry_regions_are_16_byte_aligned(cuda_lib, dk, B, R, Hq, G):
    """The carry a deferred call writes: u [B][H_v d_v/DVS][R][DVS], k^
    [B][H_qk][R][d_k], exp(g) [B][H_v][R4]; region starts and every item's
    run are 16-byte aligned, and gdn_carry_bytes is their sum."""
    Hv, dv = Hq * G, dvs(dk) * 2
    slices = dv // dvs(dk)
    u = B * R * Hv * dv
    k = B * R * Hq * dk
    a = B * Hv * round4(R)
    for off in (u, u + k, u + k + a):
        assert off % 4 == 0
    for b in range(B):
        for hs in range(Hv * slices):
            assert ((b * Hv * slices + hs) * R * dvs(dk)) % 4 == 0
        for hq in range(Hq):
            assert ((b * Hq + hq) * R * dk) % 4 == 0
        for h in range(Hv):
            assert ((b * Hv + h) * round4(R)) % 4 == 0
    args = cuda_lib.GdnArgs(B=B, R=R, H_qk=Hq, H_v=Hv, d_k=dk, d_v=dv, W=4, pool_slots=1,
                            in_dtype=cuda_lib.BF16, scale=1.0, l2_eps=1e-6, flags=0)
    assert cuda_lib.carry_bytes(args) == 4 * (u + k + a)


@pytest.mark.parametrize("elem,vv", [(2, 4), (2, 2), (2, 1), (4, 4), (4, 2), (4, 1)])
def test_prologue_value_chunks_are_aligned(elem, vv):
    """The prologue's value blocks load VV consecutive channels per row as
    one chunk (8 bytes for four bf16, 16 for four fp32): every chunk of x,
    the conv window and the taps starts on a multiple of its own size."""
    chunk = elem * vv
    for Hq, dk, Hv, dv in ((2, 16, 4, 16), (16, 128, 32, 128), (16, 128, 64, 128), (4, 64, 8, 64)):
        C = 2 * Hq * dk + Hv * dv
        for v0 in range(0, Hv * dv, vv):
            cv = 2 * Hq * dk + v0
            for row in range(3):
                assert ((row * C + cv) * elem) % chunk == 0       # x rows
            assert (cv * 4 * elem) % chunk == 0                    # taps [C][4]
            for slot in range(3):
                assert ((slot * C + cv) * 3 * elem) % min(chunk, 8 if elem == 2 else 16) == 0  # window [P][C][3]
