"""moe_permute_static_scratch, the permutation for callers that cannot
allocate device memory (a plugin handed only its input and output buffers, a
serving loop whose memory is fixed at start-up): its scratch is a fixed array
inside the library instead of a caller workspace.

Checked through the C ABI against moe_permute on the same inputs, on two
calls in a row (the second smaller, so stale scratch from the first would
show), bit for bit as every permutation test here; and sizes beyond the fixed
limit are refused on the host.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import oracle
from gpu_common import require_gpu

pytestmark = pytest.mark.gpu


def _idx(rng, T, E, k):
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


def test_static_scratch_permute_matches_workspace_permute():
    torch = require_gpu()
    from block_fp8_expert_gb300 import _lib
    L = _lib.lib()
    rng = np.random.default_rng(2024)
    for T, E, k in [(4096, 128, 8), (300, 512, 10)]:
        idx = torch.from_numpy(_idx(rng, T, E, k)).cuda()
        d = _lib.dims(T, 256, 128, E, k)
        P = T * k
        ws = torch.empty(_lib.workspace_bytes(d), dtype=torch.uint8, device="cuda")
        outs = []
        for _ in range(2):
            outs.append((torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
                         torch.full((P,), -7, dtype=torch.int32, device="cuda"),
                         torch.full((P,), -7, dtype=torch.int32, device="cuda")))
        _lib.moe_permute(idx, d, *outs[0], ws)
        st = L.moe_permute_static_scratch(idx.data_ptr(), d, outs[1][0].data_ptr(),
                                          outs[1][1].data_ptr(), outs[1][2].data_ptr(),
                                          torch.cuda.current_stream().cuda_stream)
        assert st == _lib.MOE_OK, L.moe_last_error_message()
        torch.cuda.synchronize()
        for a, b in zip(*outs):
            assert torch.equal(a, b)
        r_off, r_rt, r_tsr = oracle.permute(idx.cpu().numpy(), E)
        assert np.array_equal(outs[1][0].cpu().numpy(), r_off)
        assert np.array_equal(outs[1][1].cpu().numpy(), r_rt)
        assert np.array_equal(outs[1][2].cpu().numpy(), r_tsr)


def test_static_scratch_permute_refuses_sizes_beyond_its_limit():
    require_gpu()
    from block_fp8_expert_gb300 import _lib
    L = _lib.lib()
    for d in (_lib.dims(8193, 256, 128, 128, 8),   # T*k = 65544 > 65536
              _lib.dims(8, 256, 128, 1024, 8)):    # E > 512
        st = L.moe_permute_static_scratch(0x1000, d, 0x2000, 0x3000, 0x4000, None)
        assert st == _lib.MOE_ERR_UNSUPPORTED
        assert b"use moe_permute" in L.moe_last_error_message() or b"E <= 512" in \
            L.moe_last_error_message()


def test_static_scratch_bad_index_is_readable():
    """An expert index outside [0, E) gives its pair no row, as moe_permute
    does, and its status bit in the fixed array is read back through
    moe_read_device_status with no workspace; a clean call clears it."""
    torch = require_gpu()
    from block_fp8_expert_gb300 import _lib
    L = _lib.lib()
    T, E, k = 4, 16, 2
    d = _lib.dims(T, 256, 128, E, k)
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    rt = torch.empty(T * k, dtype=torch.int32, device="cuda")
    tsr = torch.empty(T * k, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for idx, expect in (([[0, 1], [2, 16], [-1, 3], [4, 5]], _lib.MOE_DEV_BAD_EXPERT_INDEX),
                        ([[0, 1], [2, 3], [4, 5], [6, 7]], 0)):
        ti = torch.tensor(idx, dtype=torch.int32, device="cuda")
        st = L.moe_permute_static_scratch(ti.data_ptr(), d, off.data_ptr(), rt.data_ptr(),
                                          tsr.data_ptr(), stream)
        assert st == _lib.MOE_OK, L.moe_last_error_message()
        v = ctypes.c_int32(-1)
        st = L.moe_read_device_status(None, ctypes.byref(v), stream)
        assert v.value == expect
        assert st == (_lib.MOE_ERR_DEVICE_STATUS if expect else _lib.MOE_OK)
        if expect:
            t = tsr.cpu().numpy()
            assert t[3] == -1 and t[4] == -1
            assert off.cpu().numpy()[-1] == 6
