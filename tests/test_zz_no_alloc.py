"""moe_permute_noalloc against moe_permute, through the C ABI.

moe_permute_noalloc serves callers that may not allocate device memory (a
plugin inside a framework that owns every device buffer, an allocator's own
start-up code): it keeps its counting-sort scratch in a fixed array inside
the library instead of taking a workspace.  Its outputs must equal
moe_permute's bit for bit (index and copy work), on consecutive calls with
different sizes, since the calls share that array and it keeps the previous
call's contents.

This file is collected last so that a run stopping at the first failure has
already run every other test.  It also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import moe_lora_expert_gb300 as m

MAX_SLOTS = 65536   # MOE_NOALLOC_MAX_SLOTS in include/moe_lora.h


def _lib():
    import os
    if not os.path.exists(m.LIB_PATH):
        from moe_lora_expert_gb300 import _build
        _build.build()
    return m.lib()


def test_noalloc_rejects_sizes_beyond_its_limit_on_host():
    lib = _lib()
    fake = 1 << 20
    # T * top_k = 65537 > limit: rejected before anything is enqueued (no GPU needed)
    assert lib.moe_permute_noalloc(fake, 65537, 1, 8, None, 0, fake, fake, fake, None, None,
                                   None) == m.MOE_ERR_UNSUPPORTED
    assert lib.moe_permute_noalloc(fake, 8193, 8, 128, None, 0, fake, fake, fake, None, None,
                                   None) == m.MOE_ERR_UNSUPPORTED
    assert lib.moe_permute_noalloc(fake, 4, 2, 1025, None, 0, fake, fake, fake, None, None,
                                   None) == m.MOE_ERR_UNSUPPORTED
    assert lib.moe_permute_noalloc(fake, 4, 2, 8, None, 0, None, fake, fake, None, None,
                                   None) == m.MOE_ERR_NULL


def _run_both(lib, torch, ids_np, E, hidden_np):
    """Call moe_permute (with a workspace) and moe_permute_noalloc on the same input."""
    dev = torch.device("cuda:0")
    T, k = ids_np.shape
    H = hidden_np.shape[1]
    ids = torch.from_numpy(ids_np).to(dev)
    hidden = torch.from_numpy(hidden_np.view(np.int16)).to(dev).view(torch.bfloat16)
    stream = torch.cuda.current_stream().cuda_stream
    outs = []
    for noalloc in (False, True):
        off = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
        e2p = torch.full((T * k,), -7, dtype=torch.int32, device=dev)
        p2e = torch.full((T * k,), -7, dtype=torch.int32, device=dev)
        xp = torch.zeros((T * k, H), dtype=torch.bfloat16, device=dev)
        if noalloc:
            status = torch.full((1,), 123, dtype=torch.int32, device=dev)
            rc = lib.moe_permute_noalloc(ids.data_ptr(), T, k, E, hidden.data_ptr(), H,
                                         off.data_ptr(), e2p.data_ptr(), p2e.data_ptr(),
                                         xp.data_ptr(), status.data_ptr(), stream)
            assert rc == m.MOE_OK, m.status_string(rc)
            torch.cuda.synchronize()
            st = int(status.item())
        else:
            ws = torch.empty(lib.moe_permute_workspace_size(T, k, E), dtype=torch.uint8, device=dev)
            rc = lib.moe_permute(ids.data_ptr(), T, k, E, hidden.data_ptr(), H, off.data_ptr(),
                                 e2p.data_ptr(), p2e.data_ptr(), xp.data_ptr(), ws.data_ptr(),
                                 ws.numel(), stream)
            assert rc == m.MOE_OK, m.status_string(rc)
            st = m.moe_read_device_status(ws)
        outs.append((off.cpu().numpy(), e2p.cpu().numpy(), p2e.cpu().numpy(),
                     xp.view(torch.int16).cpu().numpy(), st))
    return outs


@pytest.mark.gpu
def test_noalloc_matches_moe_permute_on_consecutive_calls():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _lib()
    rng = np.random.default_rng(2024)
    cases = [
        # a large multi-chunk call first, then a small one with fewer experts: the
        # second must not see the first call's counts left in the shared array
        (4096, 8, 128, 2048, False),
        (300, 8, 37, 72, True),
    ]
    for T, k, E, H, with_bad_id in cases:
        ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        if with_bad_id:
            ids[5, 1] = E + 3      # invalid id: dropped and reported in the status word
            ids[9, 0] = -1         # not routed
        hidden = rng.standard_normal((T, H)).astype(np.float32)
        hidden_bits = (hidden.view(np.uint32) >> 16).astype(np.uint16)
        ref, got = _run_both(lib, torch, ids, E, hidden_bits)
        for name, a, b in zip(["expert_offsets", "expanded_to_permuted", "permuted_to_expanded",
                               "permuted_hidden"], ref[:4], got[:4]):
            assert np.array_equal(a, b), f"T={T} E={E}: {name} differs"
        expect_status = m.MOE_ERR_BAD_EXPERT_ID if with_bad_id else m.MOE_OK
        assert ref[4] == expect_status and got[4] == expect_status, (ref[4], got[4])
