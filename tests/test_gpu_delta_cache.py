"""The delta cache on a device arena: asynchronous loads from pinned host
memory, requests that arrive while a load is in flight sharing it, and the
grouped linear reading its variants' signs and α straight from cache slots.

Page "BitDelta: serving 14 Zen models from one GPU cluster", section
"Infrastructure details"."""
import numpy as np
import pytest
import torch

import bit_weight_delta_gb300 as bd
import synth
import synth.device as sd

pytestmark = pytest.mark.gpu


def _cache(n_slots, slot_bytes, pin=0):
    arena = torch.empty(n_slots * slot_bytes, dtype=torch.uint8, device="cuda")
    return bd.DeltaCache(arena, slot_bytes, pin_top_k=pin)


def test_device_load_matches_the_host_bytes():
    cache = _cache(2, 1 << 20)
    host = torch.randint(0, 256, (1_000_000,), dtype=torch.uint8).pin_memory()
    cache.register(0, host)
    view = cache.acquire(0)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(view.cpu(), host)
    cache.release(0)
    cache.close()


def test_requests_during_a_load_share_it():
    slot = 256 << 20
    cache = _cache(2, slot)
    host = torch.empty(slot, dtype=torch.uint8).pin_memory()
    host.fill_(7)
    cache.register(5, host)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    a = cache.acquire(5, s1)     # starts the 256 MB copy
    b = cache.acquire(5, s2)     # arrives while it is in flight
    st = cache.stats()
    assert st["loads"] == 1 and st["queued_behind_load"] == 1
    assert a.data_ptr() == b.data_ptr()
    # both streams were made to wait for the one load
    with torch.cuda.stream(s2):
        total = b.to(torch.int64).sum()
    s2.synchronize()
    assert int(total) == 7 * slot
    cache.release(5, s1)
    cache.release(5, s2)
    cache.close()


def test_grouped_linear_on_cached_deltas_matches_direct_tensors():
    d_out, d_in, n_var, seed = 1024, 2048, 5, 21
    wb = sd.normal_bf16((d_out, d_in), seed, 1, 0.02)
    scales = synth.variant_scales(seed, n_var)
    packs, alphas, blobs = [], [], []
    pbytes = d_out * d_in // 8
    for v in range(n_var):
        wf = sd.finetuned_bf16(wb, seed, 10 + v, float(scales[v]))
        p, a = bd.bitdelta_compress(wb, wf, per_row=True)
        packs.append(p)
        alphas.append(a)
        # one blob per variant: packed signs, then α (fp32, 256-byte aligned offset)
        blob = torch.zeros(pbytes + 4 * d_out, dtype=torch.uint8)
        blob[:pbytes] = p.cpu().view(-1)
        blob[pbytes:] = a.cpu().view(torch.uint8)
        blobs.append(blob.pin_memory())
    off, var = synth.segments(seed, [1, 3, 40, 1, 2, 300, 1, 7], n_var)
    x = sd.normal_bf16((int(off[-1]), d_in), seed, 99)
    t_off, t_var = torch.from_numpy(off).cuda(), torch.from_numpy(var).cuda()
    pt, at = bd.variant_tables(packs, alphas, "cuda")
    y_direct = bd.bitdelta_linear_grouped(x, t_off, t_var, wb, pt, at, n_var=n_var,
                                          max_seg_len=300, per_row=True)
    # three slots for five variants: loads, evictions and reuse along the way
    slot = ((pbytes + 4 * d_out + 255) // 256) * 256
    cache = _cache(3, slot, pin=1)
    for v in range(n_var):
        cache.register(v + 1, blobs[v])
    y_cached = torch.empty_like(y_direct)
    for round_ in range(2):
        for vs in ((1, 2, 3), (4, 5, 1)):
            views = {v: cache.acquire(v) for v in vs}
            cp = [views[v][:pbytes] if v in views else packs[v - 1] for v in range(1, n_var + 1)]
            ca = [views[v][pbytes:].view(torch.float32) if v in views else alphas[v - 1]
                  for v in range(1, n_var + 1)]
            pt2, at2 = bd.variant_tables(cp, ca, "cuda")
            bd.bitdelta_linear_grouped(x, t_off, t_var, wb, pt2, at2, n_var=n_var,
                                       max_seg_len=300, per_row=True, out=y_cached)
            for v in vs:
                cache.release(v)
            torch.cuda.current_stream().synchronize()
            assert torch.equal(y_cached, y_direct), f"round {round_}, variants {vs}"
    st = cache.stats()
    assert st["loads"] >= 5 and st["evictions"] >= 2
    assert bd.bitdelta_check_error() == 0
    cache.close()
