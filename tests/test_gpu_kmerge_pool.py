"""The K-Merge pool driven by the GPU similarity kernel: three adapters fill
the budget B, a fourth that is a light edit of adapter 1 overflows it, the
pool asks for similarities, bitdelta_sign_similarity computes them against
the three stored entries, and the merge goes to the entry the oracle's
cosines rank first (page "BitDelta: serving 14 Zen models from one GPU
cluster", section "K-Merge": steps 1-2 and the budget-B paragraph)."""
import numpy as np
import pytest
import torch

import bit_weight_delta_gb300 as bd
import oracle
import synth
from gpu_util import to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def test_pool_merges_the_overflowing_adapter_into_the_most_similar_entry():
    torch.cuda.set_device(0)
    d_out, d_in = 512, 1024
    wb = synth.base_weight(71, d_out, d_in)
    fts = [synth.finetuned_weight(71, wb, b=1e-3 * (1 + a), stream=300 + a) for a in range(3)]
    edit = fts[1].copy()
    rng = np.random.default_rng(71)
    idx = rng.integers(0, edit.size, edit.size // 50)
    edit.flat[idx] = synth.finetuned_weight(72, wb, b=2e-3, stream=9).flat[idx]
    fts.append(edit)
    wb_d = to_dev_bf16(wb)
    comp = [bd.bitdelta_compress(wb_d, to_dev_bf16(f), per_row=True) for f in fts]
    nbytes = d_out * d_in // 8 + 4 * d_out
    pool = bd.KMergePool(3 * nbytes)
    entries = []
    for a in range(3):
        act, e = pool.request_on_device(a, nbytes, comp[a][0], comp[a][1], [], [])[:2]
        assert (act, e) == ("store", a)
        entries.append(comp[a])
    act, target, cos = pool.request_on_device(3, nbytes, comp[3][0], comp[3][1],
                                              [p for p, _ in entries], [al for _, al in entries])
    assert bd.bitdelta_check_error() == 0
    ref = []
    for p, al in entries:
        ref.append(oracle.sign_cosine(comp[3][0].cpu().numpy(), comp[3][1].cpu().numpy(),
                                      p.cpu().numpy(), al.cpu().numpy(), True)[0])
    ref = np.array(ref)
    assert np.abs(cos.numpy() - ref).max() <= 1e-9
    assert act == "merge" and target == int(np.argmax(ref)) == 1
    pool.commit(3, target, True, nbytes)
    assert pool.entry_of(3) == 1 and pool.entry_info(1) == (nbytes, 2)
    st = pool.stats()
    assert st["used_bytes"] == 3 * nbytes <= st["budget_bytes"]
    pool.close()
