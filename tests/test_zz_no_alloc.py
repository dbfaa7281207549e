"""mm_align_noalloc, the grouping entry point for callers that cannot
allocate device memory (a serving engine whose pool already owns the device,
or code where a cudaMalloc is not allowed). It keeps its per-block counts in a
fixed device array instead of the library's workspace, so it must give the
same result as mm_align: checked bit for bit (the output is integer work) on
two calls in a row that both use that array, called through the C ABI, and on
the paths that need no scratch at all (no tokens, the bitmask grouping up to
64 tokens, the one-block grouping up to 1024 tokens) with and without the
optional counts output. A call on a size mm_align has not run yet must leave
the device's free memory unchanged.

This file is collected last so that a run stopping at its first failure has
run every other test before it."""
import numpy as np
import pytest
import torch

import mixture_experts_layer_mm_gb300 as mm

pytestmark = pytest.mark.gpu


def _ids(seed, T, E, k):
    keys = np.random.default_rng(seed).random((T, E))
    ids = np.sort(np.argsort(keys, axis=1)[:, :k], axis=1).astype(np.int32)
    return torch.from_numpy(ids.reshape(T, k)).cuda()


def _outputs(T, E, k, bm, with_counts=True):
    cap = mm.mm_align_capacity(T, k, E, bm)
    s = torch.full((cap,), -7, dtype=torch.int32, device="cuda")
    off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((E,), -7, dtype=torch.int32, device="cuda") if with_counts else None
    return s, off, cnt


def _noalloc(ids, T, E, k, bm, s, off, cnt):
    L = mm.lib()
    rc = L.mm_align_noalloc(ids.data_ptr() if T > 0 else None, T, k, E, bm, s.data_ptr(),
                            off.data_ptr(), None if cnt is None else cnt.data_ptr(),
                            torch.cuda.current_stream().cuda_stream)
    assert rc == mm.MM_OK, mm.status_string(rc)


def test_no_alloc_align_matches_mm_align(mmlib):
    # Two calls in a row on different inputs, both large enough that the
    # fixed scratch array is used; the second sees the first call's leftovers.
    for seed, (T, E, k, bm) in enumerate([(16384, 128, 8, 16), (5000, 256, 6, 64)]):
        ids = _ids(seed, T, E, k)
        s_ref, off_ref, cnt_ref = mm.mm_align(ids, E, bm)
        s, off, cnt = _outputs(T, E, k, bm)
        _noalloc(ids, T, E, k, bm, s, off, cnt)
        torch.cuda.synchronize()
        assert mm.mm_poll_device_status() == mm.MM_OK
        assert torch.equal(off, off_ref)
        assert torch.equal(cnt, cnt_ref)
        assert torch.equal(s, s_ref)


@pytest.mark.parametrize("T,E,k,bm,with_counts", [
    (0, 8, 2, 16, True),        # no tokens: empty segments, sentinels only
    (64, 128, 8, 16, True),     # the bitmask grouping
    (64, 128, 8, 16, False),    # ... without the counts output
    (1024, 64, 8, 32, True),    # the one-block grouping at its largest size
    (1024, 64, 8, 32, False),
])
def test_no_alloc_align_small_paths(mmlib, T, E, k, bm, with_counts):
    ids = _ids(100 + T, T, E, k)
    s_ref, off_ref, cnt_ref = _outputs(T, E, k, bm)
    mm.mm_align(ids, E, bm, sorted_token_ids=s_ref, expert_offsets=off_ref,
                expert_counts=cnt_ref)
    s, off, cnt = _outputs(T, E, k, bm, with_counts)
    _noalloc(ids, T, E, k, bm, s, off, cnt)
    torch.cuda.synchronize()
    assert mm.mm_poll_device_status() == mm.MM_OK
    assert torch.equal(off, off_ref)
    assert torch.equal(s, s_ref)
    if with_counts:
        assert torch.equal(cnt, cnt_ref)


def test_no_alloc_align_allocates_nothing(mmlib):
    # Warm-up on another size first, so that the kernels' first launch (and
    # the one-time address look-up) has happened before memory is measured.
    E, k, bm = 96, 8, 16
    ids_w = _ids(7, 3000, E, k)
    _noalloc(ids_w, 3000, E, k, bm, *_outputs(3000, E, k, bm))
    torch.cuda.synchronize()
    T = 40000  # ceil(40000 / 256) * 96 = 15072 counts: a size no other test groups
    ids = _ids(8, T, E, k)
    s, off, cnt = _outputs(T, E, k, bm)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    _noalloc(ids, T, E, k, bm, s, off, cnt)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
    assert mm.mm_poll_device_status() == mm.MM_OK
    s_ref, off_ref, cnt_ref = mm.mm_align(ids, E, bm)
    assert torch.equal(off, off_ref) and torch.equal(cnt, cnt_ref) and torch.equal(s, s_ref)


def test_no_alloc_align_rejects_sizes_beyond_its_array(mmlib):
    L = mm.lib()
    # ceil(70000 / 256) * 128 experts = 35072 ints > the 32768 the array holds
    rc = L.mm_align_noalloc(16, 70000, 8, 128, 16, 16, 16, None, None)
    assert rc == mm.MM_ERR_UNSUPPORTED
