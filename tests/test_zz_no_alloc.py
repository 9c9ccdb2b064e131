"""The allocation-free fused entry point, for callers that cannot give the
library device memory of their own (code running during CUDA graph capture,
engines that size all device buffers once at start-up, C hosts with no device
allocator).  It runs the same kernels as the regular fused entry point on the
same inputs, with only the scratch moved into the library's fixed device
array, so it must produce the same bits, call after call (and, like the
regular one, the oracle's results); and it must refuse, before launching
anything, a call whose scratch does not fit."""
from __future__ import annotations

import pytest
import torch

import oracle
from gpu_util import bits, check_against_oracle, valid_rows
from speculative_decode_gateddeltanet_gb300.inputs import LayerSpec, make_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_static_scratch_matches_the_regular_entry_point_on_two_calls():
    from speculative_decode_gateddeltanet_gb300 import gdn

    spec = LayerSpec("no-alloc-qwen35-B16-k3", B=16, k=3, H_qk=16, H_v=32, d_k=128, d_v=128,
                     accept="uniform", pool="double")
    layer = make_layer(spec, 31)
    regular = gdn.DeviceLayer(layer, "cuda")
    static = gdn.DeviceLayer(layer, "cuda")
    valid = torch.from_numpy(valid_rows(layer)).cuda()
    for call in range(2):  # the second call starts from the first call's committed slots
        gdn.gdn_verify_commit(regular.args())
        a = static.args()
        a.work = None  # the static entry point takes no work buffer
        gdn.gdn_verify_commit_static(a)
        torch.cuda.synchronize()
        assert torch.equal(bits(static.o[valid]), bits(regular.o[valid]))
        assert torch.isnan(static.o[~valid]).all()
        assert torch.equal(bits(static.ssm_state), bits(regular.ssm_state))
        assert torch.equal(bits(static.conv_state), bits(regular.conv_state))
        assert int(static.status.item()) == 0
        if call == 0:
            check_against_oracle(layer, static, oracle.verify_commit(layer), commit=True)
        static.o.fill_(float("nan"))
        regular.o.fill_(float("nan"))


def test_static_scratch_refuses_calls_that_do_not_fit():
    from speculative_decode_gateddeltanet_gb300 import gdn

    spec = LayerSpec("too-large", B=1024, k=15, H_qk=16, H_v=64, d_k=128, d_v=128)
    a = gdn.GdnArgs(B=spec.B, R=spec.R, H_qk=spec.H_qk, H_v=spec.H_v, d_k=128, d_v=128, W=4,
                    pool_slots=spec.B, in_dtype=gdn.BF16, scale=128 ** -0.5, l2_eps=1e-6, flags=0)
    assert gdn.work_bytes(a) > gdn.STATIC_WORK_BYTES
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_verify_commit_static(a)
    assert e.value.code == gdn.ERR_TOO_LARGE
