"""Philox4x32-10 three ways: the library's device generator (gq_philox4x32_10), the oracle's C
implementation, and cuRAND's public device function curand_Philox4x32_10 (the SC'11 generator as
the CUDA toolkit ships it), called from a small kernel compiled here.  All three must agree on
random counters and keys, so neither of the project's two independent implementations can share
a mistake that the published generator does not make.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

from gpu_common import gq_module

pytestmark = pytest.mark.gpu

KERNEL = r"""
#include <cstdint>
#include <curand_kernel.h>
__global__ void k(const uint32_t* ck, uint32_t* out, int count) {
    int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= count) return;
    const uint32_t* p = ck + 6 * c;
    uint4 r = curand_Philox4x32_10(make_uint4(p[0], p[1], p[2], p[3]), make_uint2(p[4], p[5]));
    out[4 * c] = r.x; out[4 * c + 1] = r.y; out[4 * c + 2] = r.z; out[4 * c + 3] = r.w;
}
extern "C" int run(const uint32_t* ck, uint32_t* out, int count) {
    k<<<(count + 255) / 256, 256>>>(ck, out, count);
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : 1;
}
"""


@pytest.fixture(scope="module")
def curand_lib(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    d = tmp_path_factory.mktemp("curand")
    src, so = d / "philox_curand.cu", d / "libphilox_curand.so"
    src.write_text(KERNEL)
    subprocess.run([nvcc, "-gencode=arch=compute_103a,code=sm_103a", "-O2", "-shared",
                    "-Xcompiler", "-fPIC", "-o", str(so), str(src)], check=True)
    L = ctypes.CDLL(str(so))
    L.run.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    L.run.restype = ctypes.c_int
    return L


def test_three_philox_implementations_agree(oracle, curand_lib):
    import torch
    gq = gq_module()
    rng = np.random.default_rng(2023)
    count = 4096
    ck = rng.integers(0, 2**32, size=(count, 6), dtype=np.uint64).astype(np.uint32)
    ck[:8, :4] = 0                       # counter 0 and small counters
    ck[8:16, :4] = 0xFFFFFFFF            # all-ones counters
    ck[16:24, 0] = np.arange(8) | 0x80000000  # the second call's counter space
    dev = torch.from_numpy(ck.view(np.int32)).cuda()
    lib_out = gq.gq_philox4x32_10(dev).cpu().numpy().view(np.uint32)
    cu_out = torch.empty((count, 4), dtype=torch.int32, device="cuda")
    assert curand_lib.run(ctypes.c_void_p(dev.data_ptr()), ctypes.c_void_p(cu_out.data_ptr()),
                          count) == 0
    cu_out = cu_out.cpu().numpy().view(np.uint32)
    np.testing.assert_array_equal(lib_out, cu_out)
    for c in range(0, count, 97):
        want = oracle.philox4x32_10(ck[c, :4], ck[c, 4:])
        np.testing.assert_array_equal(want, cu_out[c])
