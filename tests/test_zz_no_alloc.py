"""The allocation-free counting sort (moe_permute_noalloc) against the
workspace one (moe_permute), through the C ABI, on two calls in a row.

Some callers cannot allocate device memory (an engine plugin handed no
workspace, a serving loop whose memory another allocator reserved up front,
code that must not risk an allocation's implicit device synchronisation);
this entry keeps its scratch in a fixed array inside the library instead.
Its outputs are integers, so they must equal the workspace entry's bit for
bit.  The file sorts last so that a run stopping at the first failure has
already run every other test."""

import pytest
import torch

from dropless_mixture_experts_gb300 import abi

pytestmark = pytest.mark.gpu


def _routing(T, E, k, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    scores = torch.rand(T, E, generator=g, device="cuda")
    idx = torch.argsort(scores, dim=1)[:, :k]  # k distinct experts per token
    return idx.to(torch.int32).contiguous()


def _outputs(T, E, k):
    dev = "cuda"
    return (torch.full((E,), -7, dtype=torch.int32, device=dev),
            torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
            torch.full((T * k,), -7, dtype=torch.int32, device=dev),
            torch.full((T * k,), -7, dtype=torch.int32, device=dev))


def _compare(T, E, k, idx):
    abi.load()
    stream = torch.cuda.current_stream().cuda_stream
    dims = abi.make_dims(T, 128, 128, E, k, 0, abi.MOE_BF16)
    nbytes = abi.moe_workspace_bytes(dims, abi.MOE_FWD_ONLY)
    ws = torch.empty(nbytes + 256, dtype=torch.uint8, device="cuda")
    ws_ptr = ws.data_ptr() + (-ws.data_ptr()) % 256
    ref = _outputs(T, E, k)
    abi.moe_permute(dims, idx.data_ptr(), *[t.data_ptr() for t in ref], ws_ptr, nbytes, stream)
    for call in range(2):  # the shared scratch keeps the previous call's contents
        out = _outputs(T, E, k)
        abi.moe_permute_noalloc(dims, idx.data_ptr(), *[t.data_ptr() for t in out], stream)
        torch.cuda.synchronize()
        for name, a, b in zip(("counts", "offsets", "perm", "inv_perm"), out, ref):
            assert torch.equal(a, b), (call, name)
    return ref


# (131072, 64, 8): more warp chunks than the column scan's 1024 threads (each
# thread walks two); (2^19, 256, 2): exactly the 2^19 histogram entries the
# scratch holds, the largest size accepted
@pytest.mark.parametrize("T,E,k", [(1000, 8, 2), (4097, 64, 8), (1, 4, 1), (3000, 256, 3),
                                   (131072, 64, 8), (1 << 19, 256, 2)])
def test_noalloc_permute_equals_workspace_permute(T, E, k):
    _compare(T, E, k, _routing(T, E, k, seed=T + E + k))


def test_noalloc_permute_rejected_indices_match_workspace_permute():
    # out-of-range expert indices: no sorted position (inv_perm -1) and -1
    # in perm past the sorted pairs, as the workspace sort gives them
    T, E, k = 2000, 16, 2
    idx = _routing(T, E, k, seed=11)
    idx[5, 1] = 99
    idx[17, 0] = -3
    idx[1999, 1] = E
    counts, offsets, perm, inv = _compare(T, E, k, idx)
    assert int(offsets[E]) == T * k - 3
    assert torch.all(perm[T * k - 3:] == -1)
    assert int(inv[5 * k + 1]) == -1 and int(inv[17 * k]) == -1 and int(inv[1999 * k + 1]) == -1


def test_noalloc_permute_rejects_sizes_beyond_its_scratch():
    abi.load()
    # (T*k / 512) x E above 2^19 histogram entries: rejected before any launch
    dims = abi.make_dims(1 << 20, 128, 128, 256, 2, 0, abi.MOE_BF16)
    s = abi.moe_permute_noalloc(dims, 256, 256, 256, 256, 256, None, check=False)
    assert s == abi.MOE_ERR_UNSUPPORTED
