"""Python binding of ``libgdnspec`` (the C ABI in ``include/gdnspec.h``).

Argument marshalling only: every step of the verify and commit runs in the
library's CUDA kernels.  PyTorch supplies device memory and streams.  If the
library has not been built the import fails; there is no other code path.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import torch

LIB_PATH = Path(__file__).resolve().parent / "_lib" / "libgdnspec.so"

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_MISALIGNED, ERR_LAUNCH, ERR_TOO_LARGE = 0, 1, 2, 3, 4, 5
STATIC_WORK_BYTES = 32 << 20
STATUS_BAD_SLOT, STATUS_BAD_NROWS, STATUS_BAD_ACCEPT, STATUS_TIMEOUT = 1, 2, 4, 8
STATUS_DUPLICATE_SLOT = 16  # debug/test builds only
BF16, F32 = 0, 1
FLAG_RAW_GATING = 1
FLAG_STATE_STABLE = 2  # caller's promise: nothing still running writes this call's slots, slot_ids, n_rows
REPLAY, SNAPSHOT = 0, 1

_I32, _F32, _P = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p


class GdnArgs(ctypes.Structure):
    """Mirror of ``gdn_args``."""

    _fields_ = [
        ("B", _I32), ("R", _I32), ("H_qk", _I32), ("H_v", _I32), ("d_k", _I32), ("d_v", _I32),
        ("W", _I32), ("pool_slots", _I32), ("in_dtype", _I32), ("scale", _F32), ("l2_eps", _F32),
        ("flags", _I32),
        ("x", _P), ("g", _P), ("beta", _P), ("conv_w", _P), ("conv_state", _P), ("ssm_state", _P),
        ("slot_ids", _P), ("n_rows", _P), ("accept_len", _P), ("o", _P), ("scratch_S", _P),
        ("scratch_cs", _P), ("work", _P), ("status", _P), ("A_log", _P), ("carry", _P),
    ]


class GdnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} (code {code})")


if not LIB_PATH.exists():
    raise ImportError(f"{LIB_PATH} is not built; run __graft_entry__.build() "
                      "(or python -m speculative_decode_gateddeltanet_gb300.build)")
_lib = ctypes.CDLL(str(LIB_PATH))
_lib.gdn_verify.argtypes = [ctypes.POINTER(GdnArgs), ctypes.c_int, _P]
_lib.gdn_commit.argtypes = [ctypes.POINTER(GdnArgs), ctypes.c_int, _P]
_lib.gdn_verify_commit.argtypes = [ctypes.POINTER(GdnArgs), _P]
_lib.gdn_verify_commit_static.argtypes = [ctypes.POINTER(GdnArgs), _P]
_lib.gdn_verify_commit_static.restype = ctypes.c_int
for _f in (_lib.gdn_verify, _lib.gdn_commit, _lib.gdn_verify_commit):
    _f.restype = ctypes.c_int
_lib.gdn_work_bytes.argtypes = [ctypes.POINTER(GdnArgs)]
_lib.gdn_work_bytes.restype = ctypes.c_size_t
_lib.gdn_strerror.argtypes = [ctypes.c_int]
_lib.gdn_strerror.restype = ctypes.c_char_p


class GdnAcceptArgs(ctypes.Structure):
    """Mirror of ``gdn_accept_args``."""

    _fields_ = [("B", _I32), ("R", _I32), ("V", _I32), ("in_dtype", _I32), ("logits", _P), ("drafts", _P),
                ("n_rows", _P), ("target", _P), ("accept_len", _P), ("status", _P)]


_lib.gdn_greedy_accept.argtypes = [ctypes.POINTER(GdnAcceptArgs), _P]
_lib.gdn_greedy_accept.restype = ctypes.c_int


class GdnPrevRows(ctypes.Structure):
    """Mirror of ``gdn_prev_rows``: the pending rows of a deferred commit."""

    _fields_ = [("R", _I32), ("x", _P), ("n_rows", _P), ("accept_len", _P), ("carry", _P)]


_lib.gdn_verify_deferred.argtypes = [ctypes.POINTER(GdnArgs), ctypes.POINTER(GdnPrevRows), _P]
_lib.gdn_verify_deferred.restype = ctypes.c_int
_lib.gdn_carry_bytes.argtypes = [ctypes.POINTER(GdnArgs)]
_lib.gdn_carry_bytes.restype = ctypes.c_size_t


def strerror(code: int) -> str:
    return _lib.gdn_strerror(code).decode()


def work_bytes(args: GdnArgs) -> int:
    """Bytes of scratch a call with these shapes needs (0 if the shapes are invalid)."""
    return int(_lib.gdn_work_bytes(ctypes.byref(args)))


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream or None
    return stream or None


def _check(rc: int, where: str) -> None:
    if rc != OK:
        raise GdnError(rc, where)


def gdn_verify(args: GdnArgs, mode: int = REPLAY, stream=None) -> None:
    _check(_lib.gdn_verify(ctypes.byref(args), mode, _stream(stream)), "gdn_verify")


def gdn_commit(args: GdnArgs, mode: int = REPLAY, stream=None) -> None:
    _check(_lib.gdn_commit(ctypes.byref(args), mode, _stream(stream)), "gdn_commit")


def gdn_verify_commit(args: GdnArgs, stream=None) -> None:
    _check(_lib.gdn_verify_commit(ctypes.byref(args), _stream(stream)), "gdn_verify_commit")


def gdn_verify_commit_static(args: GdnArgs, stream=None) -> None:
    """gdn_verify_commit without a work buffer (args.work is ignored): the
    library's fixed device array of STATIC_WORK_BYTES is the scratch.  For
    callers that cannot allocate device memory; see include/gdnspec.h."""
    _check(_lib.gdn_verify_commit_static(ctypes.byref(args), _stream(stream)), "gdn_verify_commit_static")


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def make_prev(*, x, n_rows, accept_len, carry) -> GdnPrevRows:
    """The previous call's pending rows for ``gdn_verify_deferred``: its x
    [B][R][C], n_rows and accept_len [B], and the carry it wrote."""
    return GdnPrevRows(R=x.shape[1], x=_ptr(x), n_rows=_ptr(n_rows), accept_len=_ptr(accept_len),
                       carry=_ptr(carry))


def carry_bytes(args: GdnArgs) -> int:
    """Bytes of carry a deferred call with these shapes writes (0 if the shapes are invalid)."""
    return int(_lib.gdn_carry_bytes(ctypes.byref(args)))


def gdn_verify_deferred(args: GdnArgs, prev: GdnPrevRows | None, stream=None) -> None:
    """Commit the previous call's accepted rows (from its carry) and verify the
    current ones in one pass (``gdn_verify_deferred``); prev None = nothing
    pending.  args.carry receives this call's carry."""
    _check(_lib.gdn_verify_deferred(ctypes.byref(args), None if prev is None else ctypes.byref(prev),
                                    _stream(stream)), "gdn_verify_deferred")


def make_args(*, x, g, beta, conv_w, conv_state, ssm_state, slot_ids, n_rows, H_qk: int,
              accept_len=None, o=None, scratch_S=None, scratch_cs=None, work=None,
              status=None, scale: float | None = None, l2_eps: float = 1e-6, A_log=None, carry=None,
              state_stable: bool = False) -> GdnArgs:
    """Fill a GdnArgs from tensors laid out as ``include/gdnspec.h`` states.

    Shapes are read from x [B][R][C], ssm_state [P][H_v][d_v][d_k] and
    conv_w [C][W]; the tensors must stay alive while the call runs.  With
    A_log given, g and beta are the raw gating projections (the raw-gating
    flag is set).  state_stable sets GDN_FLAG_STATE_STABLE: the caller
    promises that no kernel still running on the stream writes this call's
    slots, slot_ids or n_rows, so the call may fetch state early."""
    B, R, _ = x.shape
    P, H_v, d_v, d_k = ssm_state.shape
    W = conv_w.shape[1]
    if x.dtype == torch.bfloat16:
        dt = BF16
    elif x.dtype == torch.float32:
        dt = F32
    else:
        raise TypeError(f"unsupported input dtype {x.dtype}")
    return GdnArgs(
        B=B, R=R, H_qk=H_qk, H_v=H_v, d_k=d_k, d_v=d_v, W=W, pool_slots=P, in_dtype=dt,
        scale=d_k ** -0.5 if scale is None else scale, l2_eps=l2_eps,
        flags=(0 if A_log is None else FLAG_RAW_GATING) | (FLAG_STATE_STABLE if state_stable else 0),
        x=_ptr(x), g=_ptr(g), beta=_ptr(beta), conv_w=_ptr(conv_w), conv_state=_ptr(conv_state),
        ssm_state=_ptr(ssm_state), slot_ids=_ptr(slot_ids), n_rows=_ptr(n_rows),
        accept_len=_ptr(accept_len), o=_ptr(o), scratch_S=_ptr(scratch_S),
        scratch_cs=_ptr(scratch_cs), work=_ptr(work), status=_ptr(status), A_log=_ptr(A_log),
        carry=_ptr(carry))


class DeviceLayer:
    """One layer call's buffers on a CUDA device, plus the call's outputs.

    Built from a dict of CPU tensors (the layout ``inputs.make_layer`` uses).
    ``o`` is filled with NaN so rows a call must not write stay visibly
    untouched; ``status`` starts at zero; ``work`` is sized by the library.
    ``carry`` (None until set) is passed as the call's carry for deferred calls;
    ``state_stable`` (False until set) sets GDN_FLAG_STATE_STABLE on the call."""

    KEYS = ("x", "g", "beta", "conv_w", "conv_state", "ssm_state", "slot_ids", "n_rows", "accept_len")

    def __init__(self, layer: dict, device="cuda", snapshot: bool = False, scale=None,
                 l2_eps: float = 1e-6, raw_gating: bool = False):
        self.spec = layer["spec"]
        s = self.spec
        for k in self.KEYS:
            setattr(self, k, layer[k].to(device).contiguous())
        self.A_log = None
        if raw_gating:  # g and beta hold the raw projections; the library forms the gating
            self.g = layer["a_raw"].to(device).contiguous()
            self.beta = layer["b_raw"].to(device).contiguous()
            self.A_log = layer["A_log"].to(device).contiguous()
        self.o = torch.full((s.B, s.R, s.H_v, s.d_v), float("nan"), device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.scratch_S = self.scratch_cs = None
        if snapshot:
            self.scratch_S = torch.empty((s.B, s.R, s.H_v, s.d_v, s.d_k), device=device)
            self.scratch_cs = torch.empty((s.B, s.R, s.C, s.W - 1), dtype=self.x.dtype, device=device)
        self.scale, self.l2_eps = scale, l2_eps
        self.carry = None
        self.state_stable = False
        self.work = None
        self.work = torch.empty(work_bytes(self.args()) // 4, dtype=torch.float32, device=device)

    def args(self) -> GdnArgs:
        return make_args(x=self.x, g=self.g, beta=self.beta, conv_w=self.conv_w,
                         conv_state=self.conv_state, ssm_state=self.ssm_state,
                         slot_ids=self.slot_ids, n_rows=self.n_rows, accept_len=self.accept_len,
                         o=self.o, scratch_S=self.scratch_S, scratch_cs=self.scratch_cs,
                         work=self.work, status=self.status, H_qk=self.spec.H_qk,
                         scale=self.scale, l2_eps=self.l2_eps, A_log=self.A_log, carry=self.carry,
                         state_stable=self.state_stable)


def greedy_accept(logits, drafts, n_rows, target, accept_len, status=None, stream=None) -> GdnAcceptArgs:
    """Device-side greedy acceptance (``gdn_greedy_accept``): target [B][R]
    and accept_len [B] from logits [B][R][V] and drafts [B][R-1].  Returns
    the argument struct (keep the tensors alive until the stream is done)."""
    B, R, V = logits.shape
    if logits.dtype == torch.bfloat16:
        dt = BF16
    elif logits.dtype == torch.float32:
        dt = F32
    else:
        raise TypeError(f"unsupported logits dtype {logits.dtype}")
    a = GdnAcceptArgs(B=B, R=R, V=V, in_dtype=dt, logits=_ptr(logits), drafts=_ptr(drafts),
                      n_rows=_ptr(n_rows), target=_ptr(target), accept_len=_ptr(accept_len),
                      status=_ptr(status))
    _check(_lib.gdn_greedy_accept(ctypes.byref(a), _stream(stream)), "gdn_greedy_accept")
    return a
