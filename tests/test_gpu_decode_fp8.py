"""GPU parity of the one-row decode over an E4M3 KV cache (the FP8-quantized
405B model of "Context Parallelism for Scalable Million-Token Inference",
"Experimental Setup & Results"; Pass Q for decode) against the fp64 oracle on
its own dequantized inputs, through the C ABI.

The oracle quantizes each query head's row with its own scale (the kernel
does the same on the device, in the same fp32 steps, so the codes agree) and K
and V per tensor; the kernel receives the oracle's codes. One case instead
quantizes K and V with the library's own kernels, the documented workflow.

Tolerances: the scores are exact E4M3 products summed in fp32 and the sums
stay fp32, so the LSE is held to 1e-3. O differs from the exact result on the
dequantized inputs by the E4M3 rounding of P (scaled by 2^8 against each
run's exact maximum), bounded per element by oracle.fp8.pv_rounding_bound
with p_exp = 8; the check allows that bound plus 2e-4 of fp32 arithmetic plus
half a bf16 ulp of the stored output."""
import numpy as np
import pytest

import oracle
import oracle.fp8 as f8
from workloads import bf16_bits_to_f64, make_decode_inputs
from gpu_utils import assert_close, bf16_half_ulp, bf16_to_f64, cuda_ok, f32_to_f64, to_dev

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]

if cuda_ok():
    import torch
    import context_causal_attention_ring_gb300 as cpa

FP32_SLACK = 2e-4
D = 128


def _quantize_per_tensor_chunked(bits, chunk=1 << 24):
    """The oracle's per-tensor E4M3 codes and descale factor of a bf16 tensor,
    taken over slices of the flattened tensor with the whole tensor's amax
    (the codes depend only on the element and amax)."""
    flat = bits.reshape(-1)
    amax = max(float(np.abs(bf16_bits_to_f64(flat[i:i + chunk])).max())
               for i in range(0, flat.size, chunk))
    codes = np.empty(flat.size, dtype=np.uint8)
    scale = None
    for i in range(0, flat.size, chunk):
        codes[i:i + chunk], scale, _ = f8.quantize_per_tensor(
            bf16_bits_to_f64(flat[i:i + chunk]), amax=amax)
    return codes.reshape(bits.shape), scale


def _oracle_fp8(q, k, v, R):
    """O, LSE of the oracle's decode on the oracle's E4M3 inputs, the bound on
    what rounding P to E4M3 may change in O, and the K and V codes with their
    descale factors."""
    cq, sq = f8.quantize_rows(bf16_bits_to_f64(q))
    ck, sk = _quantize_per_tensor_chunked(k)
    cv, sv = _quantize_per_tensor_chunked(v)
    qd = f8.e4m3_decode(cq) * sq.astype(np.float64)[..., None]
    kd, vd = f8.dequantize(ck, sk), f8.dequantize(cv, sv)
    O_r, L_r = oracle.decode(qd, kd, vd, R)
    B, T = k.shape[0], k.shape[1]
    bound = np.stack([f8.pv_rounding_bound(qd[b:b + 1], kd[b], vd[b], [T - 1], np.arange(T),
                                           p_exp=8)[0] for b in range(B)])
    return O_r, L_r, bound, (ck, sk), (cv, sv)


def _quantize_dev(x, rows, heads, transpose):
    amax = torch.zeros(4, dtype=torch.float32, device="cuda")
    scale = torch.zeros(4, dtype=torch.float32, device="cuda")
    cpa.fp8_absmax(x, rows * heads * D, amax)
    shape = (heads, D, rows) if transpose else (rows, heads, D)
    out = torch.empty(shape, dtype=torch.uint8, device="cuda")
    cpa.fp8_quantize(x, rows, heads, D, amax, out, scale, transpose=transpose)
    return out, scale


def _run(q, k, v, R, device_quantize=False):
    B, T, Hkv = k.shape[0], k.shape[1], k.shape[2]
    Hq = q.shape[1]
    O_r, L_r, bound, (ck, sk), (cv, sv) = _oracle_fp8(q, k, v, R)
    if device_quantize:
        k8, dsk = _quantize_dev(to_dev(k.reshape(B * T, Hkv, D)), B * T, Hkv, False)
        vt8, dsv = _quantize_dev(to_dev(v.reshape(B * T, Hkv, D)), B * T, Hkv, True)
        scales = torch.stack([dsk[0], dsv[0]])
        torch.cuda.synchronize()
        assert float(dsk[0]) == sk and float(dsv[0]) == sv
    else:
        k8 = torch.from_numpy(np.ascontiguousarray(ck.reshape(B * T, Hkv, D))).cuda()
        vt8 = torch.from_numpy(np.ascontiguousarray(
            cv.reshape(B * T, Hkv, D).transpose(1, 2, 0))).cuda()
        scales = torch.tensor([sk, sv], dtype=torch.float32, device="cuda")
    qd = to_dev(q)
    o = torch.empty_like(qd)
    lse = torch.empty((Hq, B), dtype=torch.float32, device="cuda")
    ws = torch.empty(cpa.decode_workspace_size(B, R, T, Hq, Hkv, D), dtype=torch.uint8,
                     device="cuda")
    cpa.decode_fp8(qd, k8, vt8, scales, o, lse, ws, R)
    cpa.decode_sync_status()
    tag = f"decode fp8 B={B} T={T} {Hq}/{Hkv} R={R}"
    assert_close(f32_to_f64(lse), L_r, 1e-3, tag + " LSE")
    O = bf16_to_f64(o)
    err = np.abs(O - O_r)
    lim = bound + FP32_SLACK + bf16_half_ulp(O_r)
    bad = err > lim
    assert not bad.any(), (f"{tag} O: {int(bad.sum())} elements out of bound; max err "
                           f"{err.max():.3e}, max err - bound {(err - lim).max():.3e}")


@pytest.mark.parametrize("B,T,Hq,Hkv,R", [
    (2, 1024, 8, 2, 4),       # 4 heads per group, 128-key runs
    (1, 4096, 16, 1, 8),      # 16 heads per group
    (2, 768, 12, 2, 3),       # 6 heads per group, odd ring
    (3, 1536, 12, 1, 2),      # 12 heads per group
    (16, 2048, 32, 8, 8),     # 256-key runs
    (8, 4096, 32, 8, 4),      # 512-key runs
    (1, 128, 2, 2, 1),        # a single run of one tile
    (2, 8192, 64, 4, 4),      # 16 heads per group (six-slot ring), 128-key runs, 2 sequences
    (2, 1536, 48, 3, 2),      # 16 heads per group, 3 KV heads
    (4, 16384, 32, 2, 2),     # 16 heads per group, a CTA's runs cross sequences
    (2, 4096, 32, 32, 2),     # one head per group, 32 KV heads
])
def test_decode_fp8_small(B, T, Hq, Hkv, R):
    q, k, v = make_decode_inputs(B, T, Hq, Hkv, D, seed=B * 31 + R)
    _run(q, k, v, R)


@pytest.mark.parametrize("qk_scale", [0.25, 3.0])
def test_decode_fp8_score_scale(qk_scale):
    # 3.0: sharp softmax rows, where many probabilities fall into the E4M3
    # subnormals (or to zero) once scaled by 2^8
    q, k, v = make_decode_inputs(2, 2048, 16, 2, D, seed=11, qk_scale=qk_scale)
    _run(q, k, v, 4)


def test_decode_fp8_zero_and_large_query_rows():
    # a zero query row (scale 1, every code 0: uniform attention) and a row of
    # large values next to ordinary ones in the same group
    q, k, v = make_decode_inputs(2, 1024, 8, 2, D, seed=4)
    q = q.copy()
    q[0, 1] = 0
    big = (bf16_bits_to_f64(q[1, 5]) * 64.0).astype(np.float32)
    q[1, 5] = (big.view(np.uint32) >> 16).astype(np.uint16)
    _run(q, k, v, 2)


def test_decode_fp8_device_quantized():
    q, k, v = make_decode_inputs(4, 2048, 32, 8, D, seed=9)
    _run(q, k, v, 4, device_quantize=True)


def test_decode_fp8_405b_shaped_row():
    # one new row of a 405B-shaped model (128 / 8 heads) over a 131072-token
    # E4M3 cache sharded across 8 ranks
    q, k, v = make_decode_inputs(1, 131072, 128, 8, D, seed=7)
    _run(q, k, v, 8)


def test_decode_fp8_rejects_bad_shapes():
    x = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    k64 = torch.zeros((256, 1, 64), dtype=torch.uint8, device="cuda")
    k128 = torch.zeros((256, 1, D), dtype=torch.uint8, device="cuda")
    sc = torch.ones(2, dtype=torch.float32, device="cuda")
    # head_dim 64
    q = torch.zeros((1, 2, 64), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(cpa.decode_workspace_size(1, 1, 256, 2, 1, 64), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((2, 1), dtype=torch.float32, device="cuda")
    with pytest.raises(cpa.CpAttnError) as e:
        cpa.decode_fp8(q, k64, x, sc, o, lse, ws, 1)
    assert e.value.status == 3  # CP_ATTN_ERR_UNSUPPORTED
    # 64-key runs (kv_len / cp = 64)
    q = torch.zeros((1, 2, D), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(cpa.decode_workspace_size(1, 4, 256, 2, 1, D), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty_like(q)
    with pytest.raises(cpa.CpAttnError) as e:
        cpa.decode_fp8(q, k128, x, sc, o, lse, ws, 4)
    assert e.value.status == 2  # CP_ATTN_ERR_SHAPE
