"""The kernels' coarse bin over all 2^32 FP32 bit patterns against the oracle,
and the bounded-wait timeout path (a wait on a barrier nobody arrives on
records DSA_DEV_TIMEOUT and returns; the context stays usable)."""
import hashlib
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

CHUNK = 1 << 26


def _oracle_chunk_md5(start):
    from oracle import oracle as O
    return hashlib.md5(O.coarse_bin_sweep(start, CHUNK).tobytes()).hexdigest()


def test_gpu_coarse_bin_equals_oracle_on_all_2pow32_patterns():
    import dsa_sparse_attention_paged_gb300 as D
    starts = list(range(0, 1 << 32, CHUNK))
    ctx = mp.get_context("spawn")
    with ctx.Pool(min(16, os.cpu_count() or 1)) as pool:
        fut = pool.map_async(_oracle_chunk_md5, starts)
        out = torch.empty(CHUNK, dtype=torch.int16, device="cuda")
        host = torch.empty(CHUNK, dtype=torch.int16, pin_memory=True)
        gpu_md5 = []
        for s in starts:
            D.coarse_bins_range(s, CHUNK, out=out)
            host.copy_(out)
            gpu_md5.append(hashlib.md5(host.numpy().tobytes()).hexdigest())
        ref_md5 = fut.get()
    bad = [hex(s) for s, a, b in zip(starts, gpu_md5, ref_md5) if a != b]
    assert not bad, f"chunks differ: {bad[:4]}"


def test_gpu_coarse_bin_golden_values():
    import dsa_sparse_attention_paged_gb300 as D
    gold = os.path.join(os.path.dirname(__file__), "golden", "coarse_bins.txt")
    for line in open(gold):
        if line.startswith("#") or not line.strip():
            continue
        h, _v, b = line.split()[:3]
        got = int(D.coarse_bins_range(int(h, 16), 1).cpu()[0])
        assert got == int(b), (h, got, b)


def test_bounded_wait_times_out_and_reports():
    import dsa_sparse_attention_paged_gb300 as D
    ws = D.Workspace(1)
    D.wait_timeout_selftest(2_000_000, ws)   # ~1 ms at GB300 clocks
    torch.cuda.synchronize()
    assert ws.status() & D.DEV_TIMEOUT
    ws.init()
    assert ws.status() == 0
    # the context is still usable
    x = torch.arange(10, device="cuda").sum().item()
    assert x == 45


def test_closed_form_bin_key_ranges_match_the_oracle_bins():
    """The select's closed-form key range of every coarse bin: both ends are
    in the bin by the oracle's coarse_bin, the keys just outside are not, and
    the ranges tile the non-NaN keys from +inf (bin 0) down to -inf."""
    import dsa_sparse_attention_paged_gb300 as D
    from oracle import oracle as O
    kr = D.coarse_bin_key_ranges().numpy().astype(np.uint64)
    lo, hi = kr[:1024, 0], kr[:1024, 1]
    assert kr[1024, 0] > kr[1024, 1]  # past the last bin: empty

    def bins_of_keys(keys):
        keys = np.asarray(keys, dtype=np.uint64).astype(np.uint32)
        bits = np.where(keys & 0x80000000, keys ^ 0x80000000, ~keys).astype(np.uint32)
        return O.coarse_bins(bits.view(np.float32))

    T = np.arange(1024)
    assert (bins_of_keys(lo) == T).all() and (bins_of_keys(hi) == T).all()
    assert (lo <= hi).all()
    assert hi[0] == 0xFF800000 and lo[1023] == 0x007FFFFF      # +inf and -inf
    assert (lo[:-1] == hi[1:] + 1).all()                      # no gap, no overlap
    inner_below = lo[:-1] - 1                                 # the keys just below
    assert (bins_of_keys(inner_below) == T[:-1] + 1).all()
