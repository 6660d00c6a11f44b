"""The paged NVFP4 KV-cache layout of decode attention (pages of 32 tokens
per KV head: codes then E4M3 scales; a block table per sequence): packing the
oracle's logical K/V and unpacking returns them, page tables are a
permutation of the pages a sequence needs, and nothing past a sequence's
length is stored."""
import numpy as np

import layout
from block_scaled_quantized_gb300 import workloads


def test_pack_unpack_round_trip(oracle_mod):
    from oracle import resattn as ra
    B, Hkv, D, L = 3, 2, 128, 200
    _, k, _ = workloads.make_attention(B, 2 * Hkv, Hkv, D, L, seed=8)
    kc, ks = ra.kv_quantize(workloads.bf16_bits(k).reshape(-1, D))
    kc, ks = kc.reshape(B, L, Hkv, D // 2), ks.reshape(B, L, Hkv, D // 16)
    lens = np.array([200, 33, 0])
    cache, table = layout.pack_paged_cache(kc, ks, lens, rng=np.random.default_rng(0))
    assert cache.shape[1:] == (Hkv, layout.page_bytes(D)) and layout.page_bytes(D) == 32 * 72
    pages_needed = [7, 2, 0]
    used = np.concatenate([table[b, :n] for b, n in enumerate(pages_needed)])
    assert sorted(used.tolist()) == list(range(sum(pages_needed)))
    c2, s2 = layout.unpack_paged_cache(cache, table, lens, D)
    for b, n in enumerate(lens):
        np.testing.assert_array_equal(c2[b, :n], kc[b, :n])
        np.testing.assert_array_equal(s2[b, :n], ks[b, :n])
    # rows 33..63 of sequence 1's second page are not part of the cache contents
    blk = cache[table[1, 1]]
    assert not blk[:, 1 * 64:32 * 64].any() and not blk[:, 32 * 64 + 8:].any()
