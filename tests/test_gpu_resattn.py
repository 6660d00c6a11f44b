"""GPU parity of ResAttn (ResServe Sec. 4.3, Sec. 5.2) against the oracle
(oracle/resattn.py): one decode step over the paged NVFP4 KV cache through
rs_resattn_decode, max|O_gpu - O_oracle| <= 1e-3 max|O_oracle| on the fp32
output (the bar derived in tests/test_resattn_tolerance.py), with the
oracle run at the kernel's split size.  Head sizes 128 and 256, query groups
of 4, 6 and 8 heads per KV head, ragged, single-token and empty sequences,
several split counts, bf16 output, and a sequence longer than max_len
(clamped, reported in the device error word)."""
import numpy as np
import pytest
import torch

import layout
from gpu_util import DEV
from block_scaled_quantized_gb300 import rs, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_scaled_quantized_gb300 import build
    build.build()
    import oracle
    oracle.build()


def make_case(B, Hq, Hkv, D, lens, seed):
    """bf16 Q, paged K/V caches sharing one block table, and the oracle's
    logical K/V codes and scales."""
    from oracle import resattn as ra
    L = max(max(lens), 1)
    q, k, v = workloads.make_attention(B, Hq, Hkv, D, L, seed=seed)
    kc, ks = ra.kv_quantize(workloads.bf16_bits(k).reshape(-1, D))
    vc, vs = ra.kv_quantize(workloads.bf16_bits(v).reshape(-1, D))
    shp = (B, L, Hkv)
    kc, ks = kc.reshape(*shp, D // 2), ks.reshape(*shp, D // 16)
    vc, vs = vc.reshape(*shp, D // 2), vs.reshape(*shp, D // 16)
    lens = np.array(lens)
    kcache, table = layout.pack_paged_cache(kc, ks, lens, rng=np.random.default_rng(seed))
    vcache = np.zeros_like(kcache)
    for b in range(B):  # V pages follow K's block table
        for lp in range((int(lens[b]) + 31) // 32):
            t0, t1 = lp * 32, min(int(lens[b]), lp * 32 + 32)
            for h in range(Hkv):
                blk = vcache[table[b, lp], h]
                blk[:(t1 - t0) * D // 2] = vc[b, t0:t1, h].reshape(-1)
                blk[32 * D // 2:32 * D // 2 + (t1 - t0) * D // 16] = vs[b, t0:t1, h].reshape(-1)
    return q, (kc, ks, vc, vs), kcache, vcache, table


def run_gpu(q, kcache, vcache, table, lens, Hkv, max_len, out_dtype=torch.float32, alpha=None):
    B, Hq, D = q.shape
    qg = q.to(DEV)
    aq = torch.tensor([alpha], dtype=torch.float32, device=DEV)
    out = torch.full((B, Hq, D), float("nan"), dtype=out_dtype, device=DEV)
    ws = torch.empty(rs.rs_resattn_workspace_bytes(B, Hq, Hkv, D, max_len), dtype=torch.uint8, device=DEV)
    rs.rs_resattn_decode(qg, aq, torch.from_numpy(kcache).to(DEV), torch.from_numpy(vcache).to(DEV),
                         torch.from_numpy(table).to(DEV), torch.from_numpy(np.asarray(lens, np.int32)).to(DEV),
                         max_len, out, ws, Hkv)
    torch.cuda.synchronize()
    return out


CASES = [
    (2, 8, 1, 128, [700, 333]),
    (3, 32, 4, 128, [1000, 0, 129]),
    (2, 12, 2, 256, [640, 257]),
    (1, 8, 2, 128, [4096]),
    (2, 16, 4, 256, [100, 1]),
    (4, 24, 4, 128, [2048, 1500, 31, 96]),
]


@pytest.mark.parametrize("B,Hq,Hkv,D,lens", CASES)
def test_resattn_decode_parity(B, Hq, Hkv, D, lens):
    import oracle
    from oracle import resattn as ra
    q, (kc, ks, vc, vs), kcache, vcache, table = make_case(B, Hq, Hkv, D, lens, seed=B + Hq + D)
    L = max(lens)
    qb = workloads.bf16_bits(q)
    aq = float(oracle.tensor_scale(qb))
    out = run_gpu(q, kcache, vcache, table, lens, Hkv, L, alpha=aq)
    assert rs.rs_get_device_error() == 0
    st = rs.rs_resattn_split_tokens(B, Hkv, D, L, torch.cuda.get_device_properties(0).multi_processor_count)
    ref = ra.resattn_decode(qb, aq, kc, ks, vc, vs, np.array(lens), split_tokens=st)
    got = out.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    for b in range(B):
        if lens[b] == 0:
            assert np.all(got[b] == 0.0)
    err = np.abs(got - ref).max()
    assert err <= 1e-3 * np.abs(ref).max(), f"max|dO| {err:.3e} vs max|O| {np.abs(ref).max():.3e}"


def test_resattn_bf16_output():
    import oracle
    from oracle import resattn as ra
    B, Hq, Hkv, D, lens = 2, 8, 2, 128, [513, 77]
    q, (kc, ks, vc, vs), kcache, vcache, table = make_case(B, Hq, Hkv, D, lens, seed=5)
    qb = workloads.bf16_bits(q)
    aq = float(oracle.tensor_scale(qb))
    out = run_gpu(q, kcache, vcache, table, lens, Hkv, max(lens), out_dtype=torch.bfloat16, alpha=aq)
    assert rs.rs_get_device_error() == 0
    st = rs.rs_resattn_split_tokens(B, Hkv, D, max(lens), torch.cuda.get_device_properties(0).multi_processor_count)
    ref = ra.resattn_decode(qb, aq, kc, ks, vc, vs, np.array(lens), split_tokens=st)
    ref_b = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)
    got = out.float().cpu().numpy().astype(np.float64)
    bound = np.abs(ref_b) * 2.0 ** -7 + 1e-3 * np.abs(ref).max()
    assert np.all(np.abs(got - ref_b) <= bound)


def test_resattn_sequence_longer_than_max_len_is_clamped_and_reported():
    import oracle
    from oracle import resattn as ra
    B, Hq, Hkv, D = 1, 8, 2, 128
    q, (kc, ks, vc, vs), kcache, vcache, table = make_case(B, Hq, Hkv, D, [384], seed=9)
    qb = workloads.bf16_bits(q)
    aq = float(oracle.tensor_scale(qb))
    out = run_gpu(q, kcache, vcache, table, [384 + 100], Hkv, 384, alpha=aq)  # claims 100 tokens too many
    assert rs.rs_get_device_error() == rs.RS_ERR_INVALID_ARG
    st = rs.rs_resattn_split_tokens(B, Hkv, D, 384, torch.cuda.get_device_properties(0).multi_processor_count)
    ref = ra.resattn_decode(qb, aq, kc, ks, vc, vs, np.array([384]), split_tokens=st)
    got = out.cpu().numpy().astype(np.float64)
    assert np.abs(got - ref).max() <= 1e-3 * np.abs(ref).max()
