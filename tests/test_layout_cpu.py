"""Alignment of every asynchronous copy the kernel issues, for every supported
head size, input dtype, row count, group shape and CTA size: a copy must start
and end on a 16-byte boundary on both the shared and the global side.  The
formulas mirror csrc/gdn_spec.cu's `Layout`, `cluster_size` and the copies of
`issue_x` / `issue_cs` / `issue_state`; `gdn_work_bytes` is checked through
the library."""
from __future__ import annotations

import itertools

import pytest

KW, KWS = 4, 3
MAX_SMEM = 227 * 1024


def gram_floats(R):
    return (2 * R * R + 3) & ~3


def rows_per_warp(dk):
    return 8 if dk == 32 else 16


def dv_unit(dk):
    return 16 if dk == 16 else 32


def cluster_size(dk, items, es):
    for cs in (8, 4, 2):
        if items % cs == 0 and (dk // cs) * es % 16 == 0:
            return cs
    return 1


class Layout:
    """Shared-memory layout of one CTA (float offsets, then two byte stages)."""

    def __init__(self, dk, R, qs, ipc, es, D):
        nd4 = (R + 2 * R * R + 3) & ~3
        self.qk = D * dk
        self.v = self.qk + R * 2 * dk
        self.gh = self.v + ipc * R * D
        self.ab = self.gh + gram_floats(R)
        self.y = self.ab + 4 * ipc * R
        self.pd = self.y + R * 2 * qs
        self.dot = self.pd + nd4
        self.stage = self.dot + nd4
        self.st_w = R * 2 * qs * es
        self.st_cs = self.st_w + 2 * qs * KW * es
        self.st_xv = self.st_cs + 2 * qs * KWS * es
        self.st_wv = self.st_xv + R * ipc * D * es
        self.st_csv = self.st_wv + ipc * D * KW * es
        self.stage_bytes = self.st_csv + ipc * D * KWS * es
        self.bytes = 4 * self.stage + 2 * self.stage_bytes


SHAPES = list(itertools.product([16, 32, 64, 128], [2, 4], [1, 2, 3, 4, 8], [1, 2, 3, 4], [1, 2, 4, 8]))


@pytest.mark.parametrize("dk,es,units,G,nw", SHAPES)
def test_every_copy_is_16_byte_aligned(dk, es, units, G, nw):
    dv = units * dv_unit(dk)
    D = nw * rows_per_warp(dk)
    if dv % D:
        pytest.skip("slice does not divide d_v")
    slices = dv // D
    items = G * slices
    cs = cluster_size(dk, items, es)
    qs, ipc = dk // cs, items // cs
    assert qs * cs == dk and ipc * cs == items
    for Hq in (1, 3):
        Hv = Hq * G
        C = 2 * Hq * dk + Hv * dv
        for R in range(1, 17):
            L = Layout(dk, R, qs, ipc, es, D)
            if L.bytes > MAX_SMEM:
                continue  # rejected by the library's shape check
            # shared side: every region and stage piece starts on 16 bytes
            for off in (L.qk, L.v, L.gh, L.ab, L.y, L.pd, L.dot, L.stage):
                assert off % 4 == 0, (dk, R, off)
            for off in (L.st_w, L.st_cs, L.st_xv, L.st_wv, L.st_csv, L.stage_bytes):
                assert off % 16 == 0, (dk, es, R, off)
            bq, bv = qs * es, ipc * D * es
            for s in (0, 1):
                base = 4 * L.stage + s * L.stage_bytes
                for rows in range(1, R + 1):
                    for t in range(rows):
                        for dst, n in ((t * 2 * bq, bq), (t * 2 * bq + bq, bq), (L.st_xv + t * bv, bv)):
                            assert (base + dst) % 16 == 0 and n % 16 == 0
                for dst, n in ((L.st_w, KW * bq), (L.st_w + KW * bq, KW * bq), (L.st_cs, KWS * bq),
                               (L.st_cs + KWS * bq, KWS * bq), (L.st_wv, KW * bv), (L.st_csv, KWS * bv)):
                    assert (base + dst) % 16 == 0 and n % 16 == 0, (dk, es, R, dst, n)
            # global side: byte offsets from 16-byte aligned bases
            for hq, rank in itertools.product(range(Hq), range(cs)):
                chq = hq * dk + rank * qs
                chk = Hq * dk + chq
                chv = 2 * Hq * dk + hq * G * dv + rank * ipc * D
                for b, t in itertools.product(range(2), range(R)):
                    for ch in (chq, chk, chv):
                        assert ((b * R + t) * C + ch) * es % 16 == 0
                for slot in range(3):
                    for ch in (chq, chk, chv):
                        assert ch * KW * es % 16 == 0
                        assert (slot * C + ch) * KWS * es % 16 == 0
            assert (D * dk * 4) % 16 == 0  # one state slice per item


def test_cluster_shape_of_the_qwen_layer():
    # 16 q/k heads of 128, 32 value heads of 128, 8 warps (a whole head) per CTA:
    # 2 items per group, clusters of 2 CTAs with 64 q and 64 k channels each
    D = 8 * rows_per_warp(128)
    assert D == 128 and cluster_size(128, 2 * (128 // D), 2) == 2
    L = Layout(128, 4, 64, 1, 2, D)
    assert 2 * (L.bytes + 1024) <= 228 * 1024  # two CTAs fit on one SM


@pytest.mark.parametrize("dk,B,R,Hq,G", list(itertools.product([16, 128], [1, 3], [1, 3, 9, 16], [1, 2], [1, 4])))
def test_work_bytes_formula(cuda_lib, dk, B, R, Hq, G):
    Hv, dv = Hq * G, dv_unit(dk) * 2
    total = B * R * Hq * 2 * dk + B * R * Hv * dv + B * R * Hv * 4 + B * Hq * gram_floats(R)
    a = cuda_lib.GdnArgs(B=B, R=R, H_qk=Hq, H_v=Hv, d_k=dk, d_v=dv, W=4, pool_slots=1,
                         in_dtype=cuda_lib.BF16, scale=1.0, l2_eps=1e-6, flags=0)
    assert cuda_lib.work_bytes(a) == 4 * total


def test_oversized_shared_memory_is_rejected(cuda_lib):
    # 128 value heads of 256 on one q/k head: 128 items per CTA do not fit
    for nw in (1, 2, 4, 8):
        D = nw * rows_per_warp(128)
        items = 128 * (256 // D)
        cs = cluster_size(128, items, 2)
        assert Layout(128, 16, 128 // cs, items // cs, 2, D).bytes > MAX_SMEM
    a = cuda_lib.GdnArgs(B=1, R=16, H_qk=1, H_v=128, d_k=128, d_v=256, W=4, pool_slots=1,
                         in_dtype=cuda_lib.BF16, scale=1.0, l2_eps=1e-6, flags=0)
    assert cuda_lib.work_bytes(a) == 0
