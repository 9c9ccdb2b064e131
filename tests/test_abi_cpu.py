"""The C ABI without a GPU: the library loads, exports every declared entry
point, the ctypes mirror matches the C struct layout, and host-side argument
checks reject bad calls before anything is launched."""
from __future__ import annotations

import ctypes
import re
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
HEADER = ROOT / "include" / "gdnspec.h"


def declared_symbols():
    text = HEADER.read_text()
    return re.findall(r"^GDN_API\s+[\w\s\*]+?\b(\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_boundary():
    assert set(declared_symbols()) == {"gdn_verify", "gdn_commit", "gdn_verify_commit", "gdn_work_bytes",
                                      "gdn_strerror", "gdn_verify_commit_static", "gdn_greedy_accept",
                                      "gdn_verify_deferred", "gdn_carry_bytes"}


def test_library_exports_every_declared_symbol(cuda_lib):
    lib = ctypes.CDLL(str(cuda_lib.LIB_PATH))
    for name in declared_symbols():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", str(cuda_lib.LIB_PATH)], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(declared_symbols()) <= exported
    assert not any(s.startswith("_ZN7gdnspec") for s in exported), "internal symbols leak"


@pytest.mark.parametrize("mirror,cname", [("GdnArgs", "gdn_args"), ("GdnAcceptArgs", "gdn_accept_args"),
                                           ("GdnPrevRows", "gdn_prev_rows")])
def test_struct_layout_matches_header(cuda_lib, tmp_path, mirror, cname):
    cls = getattr(cuda_lib, mirror)
    fields = [f[0] for f in cls._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "gdnspec.h"\nint main(void){\n'
                   + f'printf("%zu\\n", sizeof({cname}));\n'
                   + "".join(f'printf("%zu\\n", offsetof({cname}, {f}));\n' for f in fields)
                   + "return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", str(HEADER.parent), str(src), "-o", str(exe)], check=True)
    vals = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(cls)
    for f, off in zip(fields, vals[1:]):
        assert getattr(cls, f).offset == off, f


def test_strerror_covers_codes(cuda_lib):
    for code in range(6):
        assert cuda_lib.strerror(code) and "unknown" not in cuda_lib.strerror(code)
    assert "unknown" in cuda_lib.strerror(99)


FAKE = 1 << 20  # a 16-byte aligned stand-in address; never dereferenced on these paths


def good_args(gdn, **over):
    a = gdn.GdnArgs(B=2, R=4, H_qk=16, H_v=32, d_k=128, d_v=128, W=4, pool_slots=4,
                    in_dtype=gdn.BF16, scale=128 ** -0.5, l2_eps=1e-6, flags=0)
    for f in ("x", "g", "beta", "conv_w", "conv_state", "ssm_state", "slot_ids", "n_rows",
              "accept_len", "o", "scratch_S", "scratch_cs", "work"):
        setattr(a, f, FAKE)
    for k, v in over.items():
        setattr(a, k, v)
    return a


CASES = [
    ("negative B", dict(B=-1), 1),
    ("zero rows", dict(R=0), 1),
    ("too many rows", dict(R=17), 2),
    ("conv width", dict(W=3), 2),
    ("d_k", dict(d_k=96), 2),
    ("d_v not a multiple of the block rows", dict(d_v=48), 2),
    ("H_v % H_qk", dict(H_v=24), 2),
    ("dtype", dict(in_dtype=7), 2),
    ("unknown flag", dict(flags=4), 1),
    ("raw gating without A_log", dict(flags=1), 1),
    ("misaligned A_log", dict(flags=1, A_log=FAKE + 2), 3),
    ("negative eps", dict(l2_eps=-1.0), 1),
    ("nan scale", dict(scale=float("nan")), 1),
    ("null x", dict(x=None), 1),
    ("null state", dict(ssm_state=None), 1),
    ("null o", dict(o=None), 1),
    ("null accept_len", dict(accept_len=None), 1),
    ("null work", dict(work=None), 1),
    ("misaligned work", dict(work=FAKE + 4), 3),
    ("misaligned state", dict(ssm_state=FAKE + 4), 3),
    ("misaligned o", dict(o=FAKE + 8), 3),
    ("misaligned x", dict(x=FAKE + 1), 3),
    ("misaligned status", dict(status=FAKE + 2), 3),
    ("too many requests", dict(B=70000), 2),
]


@pytest.mark.parametrize("what,over,code", CASES, ids=[c[0] for c in CASES])
def test_fused_rejects_bad_arguments(cuda_lib, what, over, code):
    a = good_args(cuda_lib, **over)
    rc = cuda_lib._lib.gdn_verify_commit(ctypes.byref(a), None)
    assert rc == code, (what, cuda_lib.strerror(rc))


def test_mode_specific_requirements(cuda_lib):
    lib, g = cuda_lib._lib, cuda_lib
    # verify needs no accept_len; snapshot verify needs scratch
    a = good_args(g, B=0, accept_len=None)
    assert lib.gdn_verify(ctypes.byref(a), g.REPLAY, None) == g.OK
    a = good_args(g, scratch_S=None)
    assert lib.gdn_verify(ctypes.byref(a), g.SNAPSHOT, None) == g.ERR_INVALID_ARG
    assert lib.gdn_verify(ctypes.byref(a), 5, None) == g.ERR_INVALID_ARG
    # snapshot commit needs scratch and accept_len, not x
    a = good_args(g, x=None, scratch_cs=None)
    assert lib.gdn_commit(ctypes.byref(a), g.SNAPSHOT, None) == g.ERR_INVALID_ARG
    a = good_args(g, B=0, x=None)
    assert lib.gdn_commit(ctypes.byref(a), g.SNAPSHOT, None) == g.OK
    # replay commit needs the work buffer; snapshot commit does not
    a = good_args(g, work=None)
    assert lib.gdn_commit(ctypes.byref(a), g.REPLAY, None) == g.ERR_INVALID_ARG
    assert lib.gdn_verify_commit(None, None) == g.ERR_INVALID_ARG


def test_empty_batch_is_a_no_op(cuda_lib):
    a = good_args(cuda_lib, B=0)
    for call in (lambda: cuda_lib._lib.gdn_verify_commit(ctypes.byref(a), None),
                 lambda: cuda_lib._lib.gdn_verify(ctypes.byref(a), 0, None),
                 lambda: cuda_lib._lib.gdn_commit(ctypes.byref(a), 0, None)):
        assert call() == cuda_lib.OK


def test_work_bytes(cuda_lib):
    a = good_args(cuda_lib)
    B, R, Hq, Hv, dk, dv = 2, 4, 16, 32, 128, 128
    assert cuda_lib.work_bytes(a) == 4 * (B * R * (2 * Hq * dk + Hv * dv + 4 * Hv) + B * Hq * ((2 * R * R + 3) // 4 * 4))
    assert cuda_lib.work_bytes(good_args(cuda_lib, d_k=96)) == 0
    assert cuda_lib._lib.gdn_work_bytes(None) == 0


def test_binding_raises_on_error(cuda_lib):
    a = good_args(cuda_lib, d_k=96)
    with pytest.raises(cuda_lib.GdnError) as e:
        cuda_lib.gdn_verify_commit(a, stream=0)
    assert e.value.code == cuda_lib.ERR_UNSUPPORTED


def test_product_never_imports_the_oracle():
    pkg = ROOT / "speculative_decode_gateddeltanet_gb300"
    for p in list(pkg.rglob("*.py")) + list(pkg.rglob("*.cu")) + list(pkg.rglob("*.h")):
        text = p.read_text()
        assert "import oracle" not in text and "from oracle" not in text, p
        assert "gdn_oracle" not in text, p


ACCEPT_CASES = [
    ("null args", None, 1),
    ("negative B", dict(B=-1), 1),
    ("zero R", dict(R=0), 1),
    ("V not a multiple of 8", dict(V=100), 2),
    ("dtype", dict(in_dtype=5), 2),
    ("null logits", dict(logits=None), 1),
    ("null drafts with R > 1", dict(drafts=None), 1),
    ("null target", dict(target=None), 1),
    ("misaligned logits", dict(logits=FAKE + 8), 3),
    ("misaligned accept_len", dict(accept_len=FAKE + 2), 3),
]


@pytest.mark.parametrize("what,over,code", ACCEPT_CASES, ids=[c[0] for c in ACCEPT_CASES])
def test_greedy_accept_rejects_bad_arguments(cuda_lib, what, over, code):
    if over is None:
        assert cuda_lib._lib.gdn_greedy_accept(None, None) == code
        return
    a = cuda_lib.GdnAcceptArgs(B=4, R=3, V=64, in_dtype=cuda_lib.BF16, logits=FAKE, drafts=FAKE, n_rows=FAKE,
                               target=FAKE, accept_len=FAKE, status=None)
    for k, v in over.items():
        setattr(a, k, v)
    assert cuda_lib._lib.gdn_greedy_accept(ctypes.byref(a), None) == code, what


def test_greedy_accept_empty_batch_is_a_no_op(cuda_lib):
    a = cuda_lib.GdnAcceptArgs(B=0, R=3, V=64, in_dtype=cuda_lib.BF16)
    assert cuda_lib._lib.gdn_greedy_accept(ctypes.byref(a), None) == cuda_lib.OK


PREV_X, PREV_CARRY = 4 << 20, 8 << 20  # the pending rows' stand-ins, clear of every FAKE range


def good_prev(gdn, **over):
    p = gdn.GdnPrevRows(R=4, x=PREV_X, n_rows=FAKE, accept_len=FAKE, carry=PREV_CARRY)
    for k, v in over.items():
        setattr(p, k, v)
    return p


DEFERRED_CASES = [
    ("zero pending rows", dict(), dict(R=0), 1),
    ("pending rows over 16", dict(), dict(R=17), 2),
    ("null pending x", dict(), dict(x=None), 1),
    ("null pending accept_len", dict(), dict(accept_len=None), 1),
    ("null pending carry", dict(), dict(carry=None), 1),
    ("misaligned pending x", dict(), dict(x=PREV_X + 2), 3),
    ("misaligned pending n_rows", dict(), dict(n_rows=FAKE + 1), 3),
    ("misaligned pending carry", dict(), dict(carry=PREV_CARRY + 4), 3),
    # a step reads the previous step's carry and rows while writing its own: no shared bytes
    ("carry out is the pending carry", dict(carry=PREV_CARRY), dict(), 1),
    ("carry out overlaps the pending carry", dict(carry=PREV_CARRY + 4096), dict(), 1),
    ("x is the pending x", dict(x=PREV_X), dict(), 1),
    ("x overlaps the pending x", dict(x=PREV_X - 65536), dict(), 1),
    ("null carry out", dict(carry=None), dict(), 1),
    ("misaligned carry out", dict(carry=FAKE + 8), dict(), 3),
    ("null o", dict(o=None), dict(), 1),
    ("null work", dict(work=None), dict(), 1),
    ("d_k", dict(d_k=96), dict(), 2),
]


@pytest.mark.parametrize("what,cur,prev,code", DEFERRED_CASES, ids=[c[0] for c in DEFERRED_CASES])
def test_deferred_rejects_bad_arguments(cuda_lib, what, cur, prev, code):
    a, p = good_args(cuda_lib, **{"carry": FAKE, **cur}), good_prev(cuda_lib, **prev)
    rc = cuda_lib._lib.gdn_verify_deferred(ctypes.byref(a), ctypes.byref(p), None)
    assert rc == code, (what, cuda_lib.strerror(rc))


def test_deferred_overlap_check_passes_distinct_buffers(cuda_lib):
    """Control for the overlap cases: the same arguments with distinct
    buffers get past every host check and fail only at the launch, which
    needs a device.  Run only where there is none (the stand-in addresses
    must never reach a real GPU)."""
    import torch

    if torch.cuda.is_available() or torch.cuda.device_count() > 0:
        pytest.skip("launch-reaching control runs only without a CUDA device")
    a, p = good_args(cuda_lib, carry=FAKE), good_prev(cuda_lib)
    assert cuda_lib._lib.gdn_verify_deferred(ctypes.byref(a), ctypes.byref(p), None) == cuda_lib.ERR_LAUNCH


def test_deferred_empty_batch_and_no_pending_rows(cuda_lib):
    lib, g = cuda_lib._lib, cuda_lib
    a = good_args(g, B=0, accept_len=None, carry=FAKE)  # the deferred call never reads accept_len
    assert lib.gdn_verify_deferred(ctypes.byref(a), ctypes.byref(good_prev(g)), None) == g.OK
    assert lib.gdn_verify_deferred(ctypes.byref(a), None, None) == g.OK
    assert lib.gdn_verify_deferred(None, None, None) == g.ERR_INVALID_ARG
    a = good_args(g, R=17, carry=FAKE)
    assert lib.gdn_verify_deferred(ctypes.byref(a), ctypes.byref(good_prev(g, R=1)), None) == g.ERR_UNSUPPORTED


def test_carry_bytes(cuda_lib):
    B, R, Hq, Hv, dk, dv = 2, 3, 16, 32, 128, 128
    a = good_args(cuda_lib, R=R)
    assert cuda_lib.carry_bytes(a) == 4 * (B * R * (Hv * dv + Hq * dk) + B * Hv * 4)
    assert cuda_lib.carry_bytes(good_args(cuda_lib, R=5)) == 4 * (B * 5 * (Hv * dv + Hq * dk) + B * Hv * 8)
    assert cuda_lib.carry_bytes(good_args(cuda_lib, d_k=96)) == 0
    assert cuda_lib._lib.gdn_carry_bytes(None) == 0


def test_status_bits_match_header(cuda_lib):
    """The binding's status constants are the header's enum values."""
    import re

    text = HEADER.read_text()
    bits = {m.group(1): int(m.group(2)) for m in re.finditer(r"GDN_(STATUS_[A-Z_]+)\s*=\s*(\d+)", text)}
    assert bits, "no status bits in the header"
    for name, value in bits.items():
        assert getattr(cuda_lib, name) == value, name
    assert len(set(bits.values())) == len(bits), "status bits overlap"
