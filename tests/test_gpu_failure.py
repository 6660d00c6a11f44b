"""Failure detection without a GPU fault: a bounded device wait that nothing
satisfies runs out, the kernel reports RS_ERR_DEVICE_TIMEOUT through the
device error word and exits, the word is cleared on reading, and the
context stays usable (a quantization afterwards is bit-exact)."""
import numpy as np
import pytest
import torch

from gpu_util import DEV, gpu_quantize, unpack
from block_scaled_quantized_gb300 import rs, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_scaled_quantized_gb300 import build
    build.build()
    import oracle
    oracle.build()


def test_bounded_wait_runs_out_and_reports():
    import oracle
    assert rs.rs_get_device_error() == rs.RS_OK
    rs.rs_debug_wait_probe(2_000_000)  # 2 ms
    assert rs.rs_get_device_error() == rs.RS_ERR_DEVICE_TIMEOUT
    assert rs.rs_get_device_error() == rs.RS_OK  # reading cleared it
    x = workloads.make_x("attn_proj_k4096", 8, K=512, seed=3)
    xb = workloads.bf16_bits(x)
    a = oracle.tensor_scale(xb)
    buf = gpu_quantize(0, x.to(DEV), torch.tensor([a], dtype=torch.float32, device=DEV), True)
    codes, sf = unpack(buf, 0, 16, 512)
    ref = oracle.quantize_residue(0, xb, a)
    np.testing.assert_array_equal(codes[0::2], ref["codes_x"])
    np.testing.assert_array_equal(codes[1::2], ref["codes_r"])
    assert rs.rs_get_device_error() == rs.RS_OK


def test_error_word_read_without_synchronization():
    """rs_get_device_error_async enqueues the read-and-clear of the error word
    behind the probe on the caller's stream and returns at once; the value is
    read from pinned host memory (and a device buffer) after an event."""
    assert rs.rs_get_device_error() == rs.RS_OK
    s = torch.cuda.Stream()
    host = torch.full((2,), -1, dtype=torch.int32).pin_memory()
    dev = torch.full((2,), -1, dtype=torch.int32, device=DEV)
    with torch.cuda.stream(s):
        rs.rs_debug_wait_probe(2_000_000, stream=s)
        rs.rs_get_device_error_async(host[0:1], stream=s)   # the timeout, then cleared
        rs.rs_get_device_error_async(dev[0:1], stream=s)    # already clear
        rs.rs_debug_wait_probe(2_000_000, stream=s)
        rs.rs_get_device_error_async(dev[1:2], stream=s)    # the second timeout
        rs.rs_get_device_error_async(host[1:2], stream=s)   # clear again
        ev = torch.cuda.Event()
        ev.record(s)
    ev.synchronize()
    assert host.tolist() == [rs.RS_ERR_DEVICE_TIMEOUT, rs.RS_OK]
    assert dev.cpu().tolist() == [rs.RS_OK, rs.RS_ERR_DEVICE_TIMEOUT]
    assert rs.rs_get_device_error() == rs.RS_OK


def test_error_word_async_argument_checks():
    import ctypes
    lib = rs.lib()
    assert lib.rs_get_device_error_async(None, None) == rs.RS_ERR_INVALID_ARG
    buf = torch.zeros(4, dtype=torch.int32, device=DEV)
    assert lib.rs_get_device_error_async(ctypes.c_void_p(buf.data_ptr() + 2), None) == rs.RS_ERR_ALIGNMENT
