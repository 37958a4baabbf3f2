"""The kernels' code conversion (the device function every kernel quantizes
with) against the oracle's encoder on every input: E4M3 and E5M2 over every
finite float32 bit pattern (all 2^32 but the NaN and infinity patterns),
INT8 over every float32 with |u| < 127.5 (the range the kernels feed it).
The oracle's side of each chunk is split across the host cores."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

CHUNK = 1 << 26               # bit patterns per comparison
INT8_LIMIT = 0x42FF0000       # bits of 127.5


@pytest.fixture(scope="module")
def taco():
    import fp8_compression_tensor_gb300 as t
    t.load_library()
    return t


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def ranges(code):
    """Bit-pattern intervals [lo, hi) to compare."""
    if code == 2:
        return [(0, INT8_LIMIT), (0x80000000, 0x80000000 + INT8_LIMIT)]
    return [(0, 0x7F800000), (0x80000000, 0xFF800000)]   # finite values of both signs


def oracle_codes(pool, threads, code, first, count):
    out = np.empty(count, dtype=np.uint8)
    part = -(-count // threads)
    jobs = [pool.submit(oracle.code_encode_bits, code, first + s, min(part, count - s), out[s:s + min(part, count - s)])
            for s in range(0, count, part)]
    for j in jobs:
        j.result()
    return out


@pytest.mark.parametrize("code", [0, 1, 2])
def test_code_conversion_matches_oracle_on_every_input(taco, code):
    threads = host_threads()
    dev = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    compared = 0
    with ThreadPoolExecutor(threads) as pool:
        for lo, hi in ranges(code):
            for first in range(lo, hi, CHUNK):
                count = min(CHUNK, hi - first)
                got = taco.selftest_encode_bits(code, first, dev[:count]).cpu().numpy()
                ref = oracle_codes(pool, threads, code, first, count)
                if not np.array_equal(got, ref):
                    bad = np.nonzero(got != ref)[0][:8]
                    pytest.fail(f"code {code}: {np.count_nonzero(got != ref)} mismatches in [{first:#x}, "
                                f"{first + count:#x}); first: "
                                + ", ".join(f"bits {first + int(i):#010x} gpu {got[i]:#04x} oracle {ref[i]:#04x}"
                                            for i in bad))
                compared += count
    expected = sum(hi - lo for lo, hi in ranges(code))
    assert compared == expected
    assert taco.device_status() == 0
