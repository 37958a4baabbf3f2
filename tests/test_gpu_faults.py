"""The device fault path, exercised without a GPU fault: a self-test kernel
waits (bounded, about 2 ms) on a barrier nothing completes, gives up like
every kernel's bounded waits do, and sets its fault bit; the host reads it
through taco_device_status(), which also clears it.  The context stays
usable: the method still runs and checks clean afterwards."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import compare_records

pytestmark = pytest.mark.gpu


def test_wait_timeout_reaches_the_host():
    import fp8_compression_tensor_gb300 as taco
    lib = taco.load_library()
    assert taco.device_status() == 0
    s = torch.cuda.Stream()
    assert lib.taco_selftest_wait_timeout(s.cuda_stream) == 0
    with pytest.raises(taco.TacoError) as err:
        taco.device_status(stream=s)
    assert err.value.status == 8
    assert taco.device_status(stream=s) == 0          # read and cleared
    bits = workloads.generate("laplace_outliers", 64, 1024, 3)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda().view(64, 1024)
    compare_records(taco.compress(x, 128).cpu().numpy(), oracle.compress(bits, 128), 128)
    assert taco.device_status() == 0


def test_flag_value_is_the_self_test_bit():
    import ctypes
    import fp8_compression_tensor_gb300 as taco
    lib = taco.load_library()
    assert lib.taco_selftest_wait_timeout(None) == 0
    flags = ctypes.c_uint32(0)
    assert lib.taco_device_status(None, ctypes.byref(flags)) == 8
    assert flags.value == 8
    assert lib.taco_device_status(None, ctypes.byref(flags)) == 0 and flags.value == 0
