"""The binding's block-list helper (argument preparation, CPU): lists built from a
boolean block mask describe the same key visibility as the mask itself."""
import numpy as np
import torch

import __graft_entry__
from oracle import block_sparse_visible


def test_lists_from_mask_round_trip():
    __graft_entry__.build()
    import exact_attention_bf16_gb300 as ea
    rng = np.random.default_rng(3)
    nq, nk = 700, 900
    nqb, nkb = -(-nq // 256), -(-nk // 128)
    for density in (0.0, 0.3, 1.0):
        mask = torch.from_numpy(rng.random((nqb, nkb)) < density)
        cnt, idx = ea.block_lists_from_mask(mask)
        assert cnt.dtype == torch.int32 and idx.dtype == torch.int32 and idx.shape[0] == nqb
        for b in range(nqb):
            listed = idx[b, :cnt[b]].tolist()
            assert listed == sorted(listed) and listed == np.flatnonzero(mask[b].numpy()).tolist()
        vis = block_sparse_visible(nq, nk, cnt.numpy(), idx.numpy())
        dense = np.repeat(np.repeat(mask.numpy(), 256, axis=0), 128, axis=1)[:nq, :nk]
        assert np.array_equal(vis, dense)
