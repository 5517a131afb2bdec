"""GPU parity of the FP8 (E4M3) path against the oracle, through the C ABI:
the quantization kernels bit for bit against the oracle's E4M3 encoder, and
the FP8 forward against fp64 attention on the oracle's own dequantized
inputs.

Tolerances (derived from the arithmetic): the scores are exact E4M3 products
summed in fp32 and the row sums stay fp32, so the LSE is held to max-abs
1e-3 like the bf16 path. O differs from the exact result by the E4M3
rounding of the probabilities that feed P V, bounded per element by
oracle.fp8.pv_rounding_bound; the check allows that bound plus 2e-4 of fp32
arithmetic plus half a bf16 ulp of the stored output.
"""
import numpy as np
import pytest

import oracle
import oracle.fp8 as f8
from workloads import WORKLOADS, Workload, bf16_bits_to_f64, make_inputs, sample_rows
from gpu_utils import DeviceRun, assert_close, bf16_half_ulp, bf16_to_f64, cuda_ok, f32_to_f64, to_dev

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]

if cuda_ok():
    import torch
    import context_causal_attention_ring_gb300 as cpa

FP32_SLACK = 2e-4
# the FP8 step scales P by 2^P_EXP before rounding it to E4M3
P_EXP = 4


def _quantize_dev(x, rows, heads, d, transpose=False):
    """Device E4M3 codes (and descale factor) of a bf16 device tensor."""
    amax = torch.zeros(4, dtype=torch.float32, device="cuda")
    scale = torch.zeros(4, dtype=torch.float32, device="cuda")
    cpa.fp8_absmax(x, rows * heads * d, amax)
    shape = (heads, d, rows) if transpose else (rows, heads, d)
    out = torch.empty(shape, dtype=torch.uint8, device="cuda")
    cpa.fp8_quantize(x, rows, heads, d, amax, out, scale, transpose=transpose)
    torch.cuda.synchronize()
    return out, float(amax[0]), float(scale[0])


@pytest.mark.parametrize("rows,heads,d,mult", [(256, 3, 128, 1.0), (128, 2, 64, 0.02),
                                               (192, 1, 128, 300.0)])
@pytest.mark.parametrize("transpose", [False, True])
def test_quantize_kernels_bit_exact(rows, heads, d, mult, transpose):
    """absmax and E4M3 quantization agree bit for bit with the oracle
    (values spread over many binades so that subnormals, ties and the
    largest code all occur)."""
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((rows, heads, d)) * np.exp2(rng.uniform(-12, 2, (rows, heads, d))) *
         mult).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)       # truncate to bf16 bits
    xv = bf16_bits_to_f64(bits)
    codes, scale, _ = f8.quantize_per_tensor(xv)
    got, amax, dscale = _quantize_dev(to_dev(bits), rows, heads, d, transpose)
    assert amax == np.float32(np.abs(xv).max())
    assert dscale == scale
    g = got.cpu().numpy()
    if transpose:
        g = g.transpose(2, 0, 1)
    assert np.array_equal(g, codes)


def test_quantize_zero_tensor():
    bits = np.zeros((64, 2, 128), dtype=np.uint16)
    got, amax, dscale = _quantize_dev(to_dev(bits), 64, 2, 128, True)
    assert amax == 0.0 and dscale == 1.0 and int(got.max()) == 0


class Fp8Run:
    """A workload quantized on the device from its rank-major bf16 tensors."""

    def __init__(self, plan, inp):
        self.base = DeviceRun(plan, inp)
        self.plan = plan
        p = plan
        self.q8, _, sq = _quantize_dev(self.base.q, p.T_q, p.Hq, p.d)
        self.k8, _, sk = _quantize_dev(self.base.k, p.T_kv, p.Hkv, p.d)
        self.vt8, _, sv = _quantize_dev(self.base.v, p.T_kv, p.Hkv, p.d, transpose=True)
        self.scales = torch.tensor([sq, sk, sv, 0.0], dtype=torch.float32, device="cuda")

    def forward(self):
        p = self.plan
        o = torch.empty((p.T_q, p.Hq, p.d), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((p.Hq, p.T_q), dtype=torch.float32, device="cuda")
        ws = torch.empty(p.workspace_size(cpa.OP_FORWARD), dtype=torch.uint8, device="cuda")
        p.forward_fp8(self.q8, self.k8, self.vt8, self.scales, o, lse, ws)
        p.sync_status()
        return o, lse, ws


def _oracle_inputs(inp):
    """The oracle's own quantization of the natural-order inputs."""
    out = []
    for x in (inp.q, inp.k, inp.v):
        codes, scale, _ = f8.quantize_per_tensor(bf16_bits_to_f64(x))
        out.append(f8.dequantize(codes, scale))
    return out


def _check_o(O, O_ref, B, what):
    err = np.abs(O - O_ref)
    lim = B + FP32_SLACK + bf16_half_ulp(O_ref)
    bad = err > lim
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements out of bound; max err "
                           f"{err.max():.3e}, max err - bound {(err - lim).max():.3e}")
    return float(err.max()), float(B.max())


def _run_and_check(w, variant="pass_kv", layout="zigzag", cu=None, chained_steps=False,
                   window=0):
    inp = make_inputs(w, with_dout=False)
    P, N = w.kv_prefix_len, w.seq_len
    plan = cpa.Plan(N, w.cp, w.n_q_heads, w.n_kv_heads, w.head_dim, layout=layout,
                    variant=variant, cu_seqlens=cu, kv_prefix_len=P, window=window)
    run = Fp8Run(plan, inp)
    if chained_steps:
        # per-step ACCUMULATE calls, chained
        plan.set_chaining(True)
        o_acc = torch.empty((plan.T_q, plan.Hq, plan.d), dtype=torch.float32, device="cuda")
        lse = torch.empty((plan.Hq, plan.T_q), dtype=torch.float32, device="cuda")
        o = torch.empty((plan.T_q, plan.Hq, plan.d), dtype=torch.bfloat16, device="cuda")
        for t in range(plan.R):
            plan.step_fwd_fp8(t, run.q8, run.k8, run.vt8, run.scales, o_acc, lse, cpa.ACCUMULATE,
                              o if t == plan.R - 1 else None)
        plan.sync_status()
    else:
        o, lse, _ = run.forward()
    qd, kd, vd = _oracle_inputs(inp)
    qpos, kpos = P + np.arange(N), np.arange(P + N)
    O_ref, L_ref = oracle.attention(qd, kd, vd, qpos, kpos, cu, window=window)
    B = f8.pv_rounding_bound(qd, kd, vd, qpos, kpos, cu, window=window, p_exp=P_EXP)
    O = run.base.to_natural_rows(bf16_to_f64(o))
    L = run.base.to_natural_rows(f32_to_f64(lse), axis=1)
    what = f"fp8 {w.name} {variant}/{layout}"
    assert_close(L, L_ref, 1e-3, what + " LSE")
    return _check_o(O, O_ref, B, what + " O")


@pytest.mark.parametrize("variant", ["pass_kv", "pass_q"])
@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("docs", [False, True])
def test_fp8_forward_variants(variant, layout, docs):
    w = Workload("fp8var", 2048, 8, 2, 128, 4)
    cu = np.array([0, 1, 130, 1000, 1023, 1024, 1500, 2048], dtype=np.int32) if docs else None
    _run_and_check(w, variant, layout, cu)


@pytest.mark.parametrize("qk_scale", [0.5, 1.0])
def test_fp8_forward_gqa_and_scale(qk_scale):
    w = Workload("fp8gqa", 4096, 16, 2, 128, 8, qk_scale=qk_scale)
    _run_and_check(w)


@pytest.mark.parametrize("variant", ["pass_kv", "pass_q"])
def test_fp8_partial_prefill(variant):
    w = Workload("fp8pp", 1024, 8, 2, 128, 2, kv_prefix_len=3072)
    _run_and_check(w, variant)


@pytest.mark.parametrize("window", [100, 1000])
def test_fp8_sliding_window_with_documents(window):
    w = Workload("fp8win", 2048, 4, 2, 128, 4)
    cu = np.array([0, 700, 1500, 2048], dtype=np.int32)
    _run_and_check(w, cu=cu, window=window)


def test_fp8_chained_per_step_calls():
    w = Workload("fp8chain", 2048, 4, 1, 128, 4)
    _run_and_check(w, chained_steps=True)


def test_fp8_step_rejects_other_head_dims():
    w = Workload("fp8d64", 1024, 2, 1, 64, 4)
    plan = cpa.Plan(w.seq_len, w.cp, w.n_q_heads, w.n_kv_heads, w.head_dim)
    x = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    sc = torch.ones(4, dtype=torch.float32, device="cuda")
    o = torch.zeros(1 << 20, dtype=torch.float32, device="cuda")
    with pytest.raises(cpa.CpAttnError) as e:
        plan.step_fwd_fp8(0, x, x, x, sc, o, o, cpa.WRITE_PARTIAL)
    assert e.value.status == 3  # CP_ATTN_ERR_UNSUPPORTED


@pytest.mark.parametrize("name", ["prefill_405b_full", "prefill_405b_partial"])
def test_fp8_prefill_405b_sampled(name):
    """The 405B-shaped prefill (128 query / 8 KV heads) in FP8, both
    orderings, at full size: O and LSE at sampled rows against the oracle on
    its own dequantized inputs (the amax of each whole tensor, the codes of
    the needed rows only)."""
    w = WORKLOADS[name]
    inp = make_inputs(w, with_dout=False)
    P, N = w.kv_prefix_len, w.seq_len
    rows = sample_rows(N, 24)
    amax_q = max(float(np.abs(bf16_bits_to_f64(inp.q[i:i + 4096])).max())
                 for i in range(0, N, 4096))
    cq, sq, _ = f8.quantize_per_tensor(bf16_bits_to_f64(inp.q[rows]), amax=amax_q)
    ck, sk, _ = f8.quantize_per_tensor(bf16_bits_to_f64(inp.k))
    kd = f8.dequantize(ck, sk)
    del ck
    cv, sv, _ = f8.quantize_per_tensor(bf16_bits_to_f64(inp.v))
    vd = f8.dequantize(cv, sv)
    del cv
    qd = f8.dequantize(cq, sq)
    qpos, kpos = P + rows, np.arange(P + N)
    O_ref, L_ref = oracle.sampled_forward(qd, kd, vd, np.arange(len(rows)), qpos, kpos)
    B = f8.pv_rounding_bound(qd, kd, vd, qpos, kpos, row_block=4, p_exp=P_EXP)
    del kd, vd
    for variant in ("pass_kv", "pass_q"):
        plan = cpa.Plan(N, w.cp, w.n_q_heads, w.n_kv_heads, w.head_dim, variant=variant,
                        kv_prefix_len=P)
        run = Fp8Run(plan, inp)
        assert float(run.scales[0]) == sq and float(run.scales[1]) == sk
        assert float(run.scales[2]) == sv
        o, lse, ws = run.forward()
        del ws
        assert_close(run.base.take(lse, rows, axis=1), L_ref, 1e-3, f"{name} {variant} LSE")
        _check_o(run.base.take(o, rows), O_ref, B, f"{name} {variant} O")
        del run, o, lse
        torch.cuda.empty_cache()


def test_fp8_pass_q_bf16_partials():
    """The E4M3 forward with bf16 Pass-Q partials against the same forward with
    fp32 partials, on the same device inputs: both compute the same fp32
    partials, so the LSE is identical and O moves only by the bf16 rounding of
    the partials (at most 2^-8 of the largest partial, itself at most max |V|)
    plus the bf16 rounding of either output."""
    w = Workload("fp8p16", 2048, 8, 2, 128, 4)
    inp = make_inputs(w, with_dout=False)
    outs = []
    for pd in ("f32", "bf16"):
        plan = cpa.Plan(w.seq_len, w.cp, w.n_q_heads, w.n_kv_heads, w.head_dim,
                        variant="pass_q", partial_dtype=pd)
        run = Fp8Run(plan, inp)
        o, lse, _ = run.forward()
        outs.append((bf16_to_f64(o), f32_to_f64(lse), run))
    (o32, l32, run), (o16, l16, _) = outs
    assert np.array_equal(l16, l32)
    _, _, vd = _oracle_inputs(inp)
    lim = 2.0 ** -8 * np.abs(vd).max() + 2 * bf16_half_ulp(np.maximum(np.abs(o32), np.abs(o16)))
    assert (np.abs(o16 - o32) <= lim).all()
    assert np.abs(o16 - o32).max() > 0   # the bf16 slots were used
