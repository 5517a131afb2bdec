"""Helpers for the GPU parity tests: moving seeded bf16 inputs to the device,
running the library through its C ABI, and comparing with the oracle."""
import numpy as np

from workloads import bf16_bits_to_f64

try:
    import torch
except Exception:  # pragma: no cover
    torch = None


def cuda_ok() -> bool:
    return torch is not None and torch.cuda.is_available()


def to_dev(bits: np.ndarray):
    """uint16 bf16 bit patterns -> torch.bfloat16 CUDA tensor (same bits)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def bf16_to_f64(t) -> np.ndarray:
    return bf16_bits_to_f64(t.view(torch.int16).cpu().numpy().view(np.uint16))


def f32_to_f64(t) -> np.ndarray:
    return t.cpu().numpy().astype(np.float64)


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the bf16 spacing at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 8)


# Flat max-abs errors of the bf16 outputs checked in this session, reported
# at the end of the run: (what, max |got - want|, elements, elements above
# the flat tolerance, largest |want| among those).
FLAT_LOG = []


def assert_close_bf16(got, want, tol=1e-2, what="", flat_below=4.0):
    """bf16 outputs against the target's flat max-abs tol.

    * Everywhere, |got - want| <= tol + half a bf16 ulp of want: the
      rounding every stored bf16 result carries, which alone reaches 2^-7 for
      |want| in [2, 4) and exceeds tol beyond 4.
    * With the target's tol (1e-2), wherever |want| < flat_below the flat
      bound |got - want| <= tol must hold. Below 4 the storage rounding is at
      most 2^-7 = 0.0078, which leaves room for the kernel's own error (P
      kept to 11 significant bits for P V). Results that were rounded to bf16
      once before (bf16 partials, whose roundings can land on neighbouring
      bf16 values on the two sides) pass flat_below=2.
    With the target's tol, the flat maximum over all elements and how many
    elements exceed tol are recorded for the session report.
    """
    err = np.abs(got - want)
    lim = tol + bf16_half_ulp(want)
    bad = err > lim
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements out of tolerance; "
                           f"max err {err.max():.3e}, max err-lim {(err - lim).max():.3e}")
    if tol >= 1e-2:
        small = np.abs(want) < flat_below
        flat = float(err[small].max()) if small.any() else 0.0
        assert flat <= tol, (f"{what}: flat max err {flat:.3e} > {tol} where "
                             f"|O| < {flat_below}")
        over = err > tol
        FLAT_LOG.append((what, float(err.max()), int(err.size), int(over.sum()),
                         float(np.abs(want[over]).max()) if over.any() else 0.0))
    return float(err.max())


def assert_close(got, want, tol, what=""):
    both_inf = np.isneginf(got) & np.isneginf(want)
    with np.errstate(invalid="ignore"):
        err = np.where(both_inf, 0.0, np.abs(got - want))
    assert np.isfinite(err).all(), f"{what}: -inf pattern differs"
    assert err.max() <= tol, f"{what}: max err {err.max():.3e} > {tol}"
    return float(err.max())


class DeviceRun:
    """Inputs of one workload on the device, in the plan's rank-major order."""

    def __init__(self, plan, inp):
        import context_causal_attention_ring_gb300 as cpa
        self.cpa = cpa
        self.plan = plan
        self.inp = inp
        q, k, v = to_dev(inp.q), to_dev(inp.k), to_dev(inp.v)
        self.q = torch.empty_like(q)
        self.k = torch.empty_like(k)
        self.v = torch.empty_like(v)
        plan.layout_apply(cpa.TENSOR_Q, cpa.TO_RANK_MAJOR, q, self.q)
        plan.layout_apply(cpa.TENSOR_KV, cpa.TO_RANK_MAJOR, k, self.k)
        plan.layout_apply(cpa.TENSOR_KV, cpa.TO_RANK_MAJOR, v, self.v)
        self.dout = None
        if inp.dout is not None:
            do = to_dev(inp.dout)
            self.dout = torch.empty_like(do)
            plan.layout_apply(cpa.TENSOR_Q, cpa.TO_RANK_MAJOR, do, self.dout)
        del q, k, v
        # natural row of each rank-major row (sequence b of a batch holds
        # positions [b L, (b + 1) L), L = prefix + new tokens)
        P = plan.kv_prefix_len
        N = plan.T_q // plan.batch
        L = plan.T_kv // plan.batch
        qpos = np.concatenate([plan.positions(cpa.TENSOR_Q, r) for r in range(plan.R)])
        b = qpos // L
        self.q_nat = b * N + (qpos - b * L - P)
        self.kv_nat = np.concatenate([plan.positions(cpa.TENSOR_KV, r) for r in range(plan.R)])

    def forward(self):
        cpa, p = self.cpa, self.plan
        o = torch.empty_like(self.q)
        lse = torch.empty((p.Hq, p.T_q), dtype=torch.float32, device="cuda")
        ws = torch.empty(p.workspace_size(cpa.OP_FORWARD), dtype=torch.uint8, device="cuda")
        p.forward(self.q, self.k, self.v, o, lse, ws)
        p.sync_status()
        return o, lse, ws

    def take_index(self, nat_rows, kind="q") -> np.ndarray:
        """Rank-major row index of each natural row."""
        nat = self.q_nat if kind == "q" else self.kv_nat
        inv = np.empty_like(nat)
        inv[nat] = np.arange(len(nat))
        return inv[np.asarray(nat_rows)].astype(np.int64)

    def take(self, t, nat_rows, kind="q", axis=0) -> np.ndarray:
        """Rows (natural indices) of a rank-major device tensor, gathered on
        the device and returned as fp64 host data."""
        idx = torch.from_numpy(self.take_index(nat_rows, kind)).to(t.device)
        g = torch.index_select(t, axis, idx)
        if g.dtype == torch.bfloat16:
            return bf16_to_f64(g.contiguous())
        return g.double().cpu().numpy()

    def to_natural_rows(self, x_rm: np.ndarray, kind="q", axis=0):
        """Reorder a host array from rank-major rows to natural rows."""
        nat = self.q_nat if kind == "q" else self.kv_nat
        out = np.empty_like(x_rm)
        idx = [slice(None)] * x_rm.ndim
        idx[axis] = nat
        out[tuple(idx)] = x_rm
        return out
