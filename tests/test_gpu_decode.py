"""GPU parity of the one-row decode over the emulated ring (kernel K8 plus
the K4 merge; Pass Q for decode, "Context Parallelism for Scalable
Million-Token Inference") against the fp64 oracle, through the C ABI. Covers
one to sixteen query heads per KV head (including group sizes that are not a
multiple of four), both head dimensions, several ring sizes and a 405B-shaped
row over 131072 keys. With head_dim 128 and key runs of 128, 256 or 512 the
tensor-core kernel (K9) computes the partials; head_dim 64 and 64-key runs
use the CUDA-core kernel (K8). K9 is a persistent grid whose CTAs each keep
one KV head and take its runs from a work counter, merging consecutive runs
of one sequence: the cases with several sequences and more runs than CTAs
cover runs that cross sequences. Tolerances: O (bf16) 1e-2 plus half a bf16
ulp, LSE 1e-3."""
import numpy as np
import pytest

import oracle
from workloads import bf16_bits_to_f64, make_decode_inputs
from gpu_utils import assert_close, assert_close_bf16, bf16_to_f64, cuda_ok, f32_to_f64, to_dev

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]

if cuda_ok():
    import torch
    import context_causal_attention_ring_gb300 as cpa


def _check(B, T, Hq, Hkv, d, R, seed, qk_scale=1.0):
    q, k, v = make_decode_inputs(B, T, Hq, Hkv, d, seed=seed, qk_scale=qk_scale)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    o = torch.empty_like(qd)
    lse = torch.empty((Hq, B), dtype=torch.float32, device="cuda")
    ws = torch.empty(cpa.decode_workspace_size(B, R, T, Hq, Hkv, d), dtype=torch.uint8,
                     device="cuda")
    cpa.decode(qd, kd, vd, o, lse, ws, R)
    cpa.decode_sync_status()
    O_r, L_r = oracle.decode(bf16_bits_to_f64(q), bf16_bits_to_f64(k), bf16_bits_to_f64(v), R)
    tag = f"decode B={B} T={T} {Hq}/{Hkv} d={d} R={R}"
    assert_close_bf16(bf16_to_f64(o), O_r, 1e-2, tag + " O")
    assert_close(f32_to_f64(lse), L_r, 1e-3, tag + " LSE")


@pytest.mark.parametrize("B,T,Hq,Hkv,d,R", [
    (2, 1024, 8, 2, 128, 4),      # 4 heads per group
    (1, 4096, 16, 1, 128, 8),     # 16 heads per group
    (3, 512, 4, 4, 64, 2),        # one head per group, d = 64
    (2, 768, 12, 2, 128, 3),      # 6 heads per group, odd ring
    (1, 64, 2, 1, 64, 1),         # a single 64-key run
    (16, 2048, 32, 8, 128, 8),    # many sequences: 256-key runs
    (2, 8192, 64, 4, 128, 4),     # 16 heads per group, 128-key runs of a 2048-key shard
    (3, 1536, 12, 1, 128, 2),     # 12 heads per group, 128-key runs of a 768-key shard
    (2, 1536, 48, 3, 128, 2),     # 16 heads per group, 3 KV heads (the grid is a multiple of 3)
    (4, 16384, 32, 2, 128, 2),    # 16 heads per group, a CTA's runs cross sequences
    (2, 4096, 32, 32, 128, 2),    # one head per group, 32 KV heads (9 CTAs per KV head)
])
def test_decode_small(B, T, Hq, Hkv, d, R):
    _check(B, T, Hq, Hkv, d, R, seed=B * 100 + R)


def test_decode_405b_shaped_row():
    # one new row of a 405B-shaped model (128 / 8 heads) over a 131072-token
    # context sharded across 8 ranks
    _check(1, 131072, 128, 8, 128, 8, seed=7)


def test_decode_rejects_bad_shapes():
    with pytest.raises(cpa.CpAttnError):
        cpa.decode_workspace_size(1, 4, 100, 8, 2, 128)       # kv_len not a multiple of 64*cp
    with pytest.raises(cpa.CpAttnError):
        cpa.decode_workspace_size(1, 1, 64, 34, 2, 128)       # 17 heads per group
