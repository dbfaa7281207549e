"""mm_align_noalloc, the grouping entry point for callers that cannot
allocate device memory (a serving engine whose pool already owns the device,
or code where a cudaMalloc is not allowed). It keeps its per-block counts in a
fixed device array instead of the library's workspace, so it must give the
same result as mm_align: checked bit for bit (the output is integer work) on
two calls in a row that both use that array, called through the C ABI.

This file is collected last so that a run stopping at its first failure has
run every other test before it."""
import ctypes

import numpy as np
import pytest
import torch

import mixture_experts_layer_mm_gb300 as mm

pytestmark = pytest.mark.gpu


def _ids(seed, T, E, k):
    keys = np.random.default_rng(seed).random((T, E))
    ids = np.sort(np.argsort(keys, axis=1)[:, :k], axis=1).astype(np.int32)
    return torch.from_numpy(ids).cuda()


def test_no_alloc_align_matches_mm_align(mmlib):
    L = mm.lib()
    stream = torch.cuda.current_stream().cuda_stream
    # Two calls in a row on different inputs, both large enough that the
    # fixed scratch array is used; the second sees the first call's leftovers.
    for seed, (T, E, k, bm) in enumerate([(16384, 128, 8, 16), (5000, 256, 6, 64)]):
        assert mm.mm_align_capacity(T, k, E, bm) > 0
        ids = _ids(seed, T, E, k)
        s_ref, off_ref, cnt_ref = mm.mm_align(ids, E, bm)
        cap = mm.mm_align_capacity(T, k, E, bm)
        s = torch.full((cap,), -7, dtype=torch.int32, device="cuda")
        off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
        cnt = torch.full((E,), -7, dtype=torch.int32, device="cuda")
        rc = L.mm_align_noalloc(ids.data_ptr(), T, k, E, bm, s.data_ptr(), off.data_ptr(),
                                cnt.data_ptr(), stream)
        assert rc == mm.MM_OK, mm.status_string(rc)
        torch.cuda.synchronize()
        assert mm.mm_poll_device_status() == mm.MM_OK
        assert torch.equal(off, off_ref)
        assert torch.equal(cnt, cnt_ref)
        assert torch.equal(s, s_ref)


def test_no_alloc_align_rejects_sizes_beyond_its_array(mmlib):
    L = mm.lib()
    # ceil(70000 / 256) * 128 experts = 35072 ints > the 32768 the array holds
    rc = L.mm_align_noalloc(16, 70000, 8, 128, 16, 16, 16, None, None)
    assert rc == mm.MM_ERR_UNSUPPORTED
