"""The bounded staging wait of the rows kernel, made to run out on the GPU.

A test-only build of the library (GDN_TEST_HOOKS, 2 ms wait limit) lets a test
name one rows-kernel item whose state copy the producer declares on its
barrier but never issues.  No copy is then in flight, the item's wait runs out
after the limit, and the CTA must set GDN_STATUS_TIMEOUT, write nothing for
that item, and leave the context usable.  Everything the other items and the
prologue write must still match the oracle."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_util import O_TOL, S_TOL, bits, check_against_oracle, valid_rows
from speculative_decode_gateddeltanet_gb300.inputs import LayerSpec, make_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hooks(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decode_gateddeltanet_gb300 import build as pkg_build

    lib = ctypes.CDLL(str(pkg_build.build_test_hooks()))
    lib.gdn_verify_commit.argtypes = [ctypes.POINTER(cuda_lib.GdnArgs), ctypes.c_void_p]
    lib.gdn_verify_commit.restype = ctypes.c_int
    lib.gdn_test_drop_state_copy.argtypes = [ctypes.c_int]
    lib.gdn_test_drop_state_copy.restype = ctypes.c_int
    yield lib
    lib.gdn_test_drop_state_copy(-1)


SPEC = LayerSpec("timeout-qwen35-B2-k3", B=2, k=3, H_qk=16, H_v=32, d_k=128, d_v=128, accept="uniform",
                 pool="double")


def test_a_wait_that_runs_out_sets_the_status_and_writes_nothing(hooks, cuda_lib):
    gdn = cuda_lib
    layer = make_layer(SPEC, 55)
    slices, dvs = SPEC.d_v // 32, 32
    # B=2 gives 256 items, one per CTA: the dropped item is the only one lost
    b, h, sl = 0, 19, 1
    item = (b * SPEC.H_v + h) * slices + sl
    assert hooks.gdn_test_drop_state_copy(item) == 0
    dev = gdn.DeviceLayer(layer, "cuda")
    assert hooks.gdn_verify_commit(ctypes.byref(dev.args()), None) == 0
    torch.cuda.synchronize()  # returns: the kernel gave up on the wait instead of spinning
    assert int(dev.status.item()) == gdn.STATUS_TIMEOUT  # and no other bit

    ref = oracle.verify_commit(layer)
    rows = slice(sl * dvs, (sl + 1) * dvs)
    o = dev.o.double().cpu().numpy()
    assert np.isnan(o[b, :, h, rows]).all(), "the timed-out item wrote o"
    valid = valid_rows(layer)
    keep = np.ones_like(o, dtype=bool)
    keep[b, :, h, rows] = False
    sel = valid[:, :, None, None] & keep
    err = float(np.abs(o[sel] - ref["o"][sel]).max() / np.abs(ref["o"][sel]).max())
    assert err <= O_TOL
    S = dev.ssm_state.cpu()
    slot = int(layer["slot_ids"][b])
    assert torch.equal(bits(S[slot, h, rows]), bits(layer["ssm_state"][slot, h, rows])), "timed-out slice written"
    want = ref["ssm_state"].copy()
    want[slot, h, rows] = layer["ssm_state"][slot, h, rows].double().numpy()  # the slice left as it was
    for bb in range(SPEC.B):
        s = int(layer["slot_ids"][bb])
        e = float(np.linalg.norm(S[s].double().numpy() - want[s]) / np.linalg.norm(want[s]))
        assert e <= S_TOL
    # the prologue commits the conv windows whatever the rows kernel did
    ref_cs = torch.from_numpy(ref["conv_state"]).to(dev.conv_state.dtype)
    assert torch.equal(bits(dev.conv_state), bits(ref_cs))

    # the context is still usable: the same call with every copy issued matches the oracle
    assert hooks.gdn_test_drop_state_copy(-1) == 0
    again = gdn.DeviceLayer(layer, "cuda")
    assert hooks.gdn_verify_commit(ctypes.byref(again.args()), None) == 0
    torch.cuda.synchronize()
    assert int(again.status.item()) == 0
    check_against_oracle(layer, again, ref, commit=True)
