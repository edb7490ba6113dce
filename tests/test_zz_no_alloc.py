"""lora_delta_fused_noalloc: the routed delta for callers that cannot allocate.

Some callers cannot call cudaMalloc on the path that applies the delta (a
memory budget fixed at start up, an allocator that refuses allocations after
warm-up, a runtime that only lends the library tensors it already owns), so
they cannot hand lora_delta_fused its scratch workspace.  The no-allocation
entry point takes that scratch from a fixed buffer inside the library.  These
tests call it through the C ABI and hold it to the existing entry point's
results and to the CPU oracle within the parity tolerance, on two calls in a
row (the second call reuses the buffer the first one left behind).  They also
check what the entry point exists for: once a first call on the device has
reserved the buffer, a call leaves the device's free memory where it was.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from lora_delta_gb300 import inputs
from tests.gpu_util import assert_close, oracle_delta

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ld():
    import __graft_entry__
    __graft_entry__.build()
    import lora_delta_gb300
    assert torch.cuda.is_available()
    return lora_delta_gb300


def _cases():
    # n > 1024 rows: the rows are clustered by slot in the scratch buffer
    a = inputs.prefill_gate_up_case(seed=91, n_tokens=3000, n_segments=12, seg_lo=16,
                                    seg_hi=700, k_in=512, widths=(1024, 776))
    b = inputs.linear_case(92, n=2500, k_in=512, widths=(1024, 776), max_loras=8,
                           max_rank=32, ranks=[32, 16, 8, 32, 24, 32, 8, 16], alpha=32.0,
                           p_none=0.1)
    return a, b


def test_noalloc_matches_fused_and_oracle_on_two_calls_in_a_row(ld, oracle):
    from lora_delta_gb300 import device_inputs as di
    assert ld.lora_noalloc_scratch_bytes() == 4 << 20
    for case in _cases():
        d = di.linear_to_device(case)
        ref = d.out0.clone()
        ld.lora_delta_fused(ref, d.x, d.seq_slot, d.pool)
        want, want_err = oracle_delta(oracle, case)
        for call in range(2):
            got = d.out0.clone()
            err = ld.new_error_word()
            ld.lora_delta_fused_noalloc(got, d.x, d.seq_slot, d.pool, err=err)
            assert ld.lora_get_error(err) == want_err == 0
            g = di.bits(got)
            assert_close(g, di.bits(ref), f"noalloc vs lora_delta_fused, call {call + 1}")
            assert_close(g, want, f"noalloc vs the oracle, call {call + 1}")
            unrouted = case.seq_slot < 0
            assert np.array_equal(g[unrouted], case.out0[unrouted])


def test_noalloc_call_leaves_free_device_memory_unchanged(ld):
    """After the warm-up call that reserves the buffer on this device, another call
    does not move the device's free memory."""
    from lora_delta_gb300 import device_inputs as di
    case = _cases()[1]
    d = di.linear_to_device(case)
    out = d.out0.clone()
    err = ld.new_error_word()
    ld.lora_delta_fused_noalloc(out, d.x, d.seq_slot, d.pool, err=err)  # warm-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    ld.lora_delta_fused_noalloc(out, d.x, d.seq_slot, d.pool, err=err)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert ld.lora_get_error(err) == 0


def test_noalloc_rejects_batches_beyond_its_buffer_and_leaves_out_unchanged(ld):
    L = ld.lib()
    w = (ctypes.c_int32 * 1)(16)
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: the size check comes first
    n = (4 << 20) // 4 + 1024
    rc = L.lora_delta_fused_noalloc(fake, 16, fake, n, 16, fake, fake, fake, None, w, 1, 16, 4,
                                    0, 1, None, None)
    assert rc == 7 and ld.status_string(rc) == "LORA_ERR_TOO_LARGE"
    # the same refusal on real tensors: nothing is enqueued, out keeps its bits
    from lora_delta_gb300 import device_inputs as di
    n = 50_000  # lora_workspace_min_size(50000, 2, 32, 8) is about 13 MB > 4 MiB
    case = inputs.linear_case(93, n=n, k_in=64, widths=(64, 32), max_loras=8, max_rank=32,
                              ranks=[32] * 8, alpha=32.0)
    d = di.linear_to_device(case)
    assert ld.lora_workspace_min_size(n, 2, 32, 8) > ld.lora_noalloc_scratch_bytes()
    out = d.out0.clone()
    with pytest.raises(ld.LoraError) as e:
        ld.lora_delta_fused_noalloc(out, d.x, d.seq_slot, d.pool)
    assert e.value.code == 7
    torch.cuda.synchronize()
    assert np.array_equal(di.bits(out), case.out0)
