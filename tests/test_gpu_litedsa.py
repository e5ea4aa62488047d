"""LiteDSA packing on the GPU against the CPU oracle (integer work: bit-exact)."""
import numpy as np
import pytest

import oracle.litedsa as ld
from indexer_topk_long_gb300 import IndexerTopK, datagen, litedsa_pack
from parity import to_device

pytestmark = pytest.mark.gpu


def _compare(idx_np, group):
    import torch
    u, lens, m = litedsa_pack(torch.from_numpy(idx_np.astype(np.int32)).cuda(), group)
    torch.cuda.synchronize()
    ru, rl, rm = ld.pack(idx_np, group)
    np.testing.assert_array_equal(lens.cpu().numpy(), rl)
    np.testing.assert_array_equal(u.cpu().numpy(), ru)
    np.testing.assert_array_equal(m.cpu().numpy().view(np.uint32), rm)
    return rl


@pytest.mark.parametrize("T,k,G", [(100, 64, 8), (37, 100, 5), (9, 2048, 8), (64, 512, 32)])
def test_random_overlapping_selections(T, k, G):
    rng = np.random.default_rng(T * k)
    pool = rng.choice(1 << 20, size=3 * k, replace=False)
    idx = np.stack([rng.choice(pool, size=k, replace=False) for _ in range(T)])
    idx[rng.random(idx.shape) < 0.05] = -1          # empty slots
    _compare(idx, G)


def test_packs_real_indexer_output():
    import torch
    inp = datagen.workload_inputs("tiny")
    op = IndexerTopK(max_T=32, max_S=8192, k=2048)
    d = to_device(inp)
    idx, _ = op(d["q"], d["w"], d["k_cache"], d["positions"], k=2048)
    torch.cuda.synchronize()
    op.close()
    lens = _compare(idx.cpu().numpy(), 8)
    # neighbouring queries share most of their keys: far fewer list entries
    assert lens.sum() < 0.5 * 32 * 2048


@pytest.mark.parametrize("T,k,G", [(24, 1024, 8), (6, 4, 3)])
def test_large_indices_use_wide_keys(T, k, G):
    """Indices of 2^24 and above take the 64-bit key path; mixed groups too."""
    rng = np.random.default_rng(7 + k)
    pool = rng.choice(np.arange((1 << 24) - 4 * k, (1 << 31) - 1, dtype=np.int64), size=3 * k, replace=False)
    idx = np.stack([rng.choice(pool, size=k, replace=False) for _ in range(T)])
    idx[: T // 2] %= (1 << 24)                       # first half of the groups: small indices only
    idx[rng.random(idx.shape) < 0.05] = -1
    _compare(idx, G)


def test_full_groups_of_16384_keys():
    """G * k = 16384 (the largest group): duplicates across all eight queries."""
    rng = np.random.default_rng(99)
    pool = rng.choice(1 << 20, size=3000, replace=False)
    idx = np.stack([rng.choice(pool, size=2048, replace=False) for _ in range(16)])
    _compare(idx, 8)
