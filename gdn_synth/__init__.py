"""Seeded synthetic inputs for the chunked gated-delta-rule prefill.

This module only draws random numbers and lays them out in memory. It holds
none of the method's arithmetic, so both the CPU oracle and the CUDA path can
be fed from it without sharing any computation.

Distributions follow the workloads the GDN prefill op is measured on
(ssm_gdn_a3.rs, `gdn_prefill_fla` problem arguments): q and k are N(0,1)
with every 128-wide head row L2-normalised, v is N(0,1), all three stored as
bf16; the log-gate g = -softplus(N(mu, sigma)) and beta = sigmoid(N(0,1)) are
fp32; the carried state is fp32 [nv, dk, dv] per sequence.

Every array is drawn from its own child stream of one numpy SeedSequence, in
the fixed order q, k, v, g, beta, h0, lengths, so changing one shape never
perturbs another array's values.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Problem",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "make_problem",
    "config_problem",
    "CONFIGS",
]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest, ties to even); returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    out = ((u + rounding) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


@dataclass
class Problem:
    """One prefill problem in the layout the C-ABI takes.

    Row r of every per-token array is token r of the packed batch: dense mode
    uses r = b*T + t, varlen mode r = cu_seqlens[s] + t.
    """

    B: int
    T: int  # dense: tokens per sequence; varlen: total packed rows
    nk: int
    nv: int
    dk: int
    dv: int
    q: np.ndarray  # uint16 bf16 bits [rows, q_stride]
    k: np.ndarray  # uint16 bf16 bits [rows, k_stride]
    v: np.ndarray  # uint16 bf16 bits [rows, v_stride]
    g: np.ndarray  # float32 [rows, g_stride]
    beta: np.ndarray  # float32 [rows, beta_stride]
    h0: np.ndarray  # float32 [B, nv, dk, dv]
    cu_seqlens: np.ndarray | None = None  # int32 [B+1] or None (dense)
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def rows(self) -> int:
        return self.q.shape[0]

    @property
    def varlen(self) -> bool:
        return self.cu_seqlens is not None

    def seq_bounds(self):
        """(start_row, length) of each sequence."""
        if self.cu_seqlens is None:
            return [(b * self.T, self.T) for b in range(self.B)]
        cu = self.cu_seqlens
        return [(int(cu[s]), int(cu[s + 1] - cu[s])) for s in range(self.B)]

    @property
    def tokens(self) -> int:
        return sum(n for _, n in self.seq_bounds())


def _softplus(x):
    return np.logaddexp(0.0, x)


def _normalised_rows(rng, rows, heads, d):
    x = rng.standard_normal((rows, heads, d), dtype=np.float32)
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True, dtype=np.float32))
    return (x / np.maximum(n, np.float32(1e-30))).astype(np.float32)


def _raw_rows(rng, rscale, rows, heads, d):
    # un-normalised rows for the fused-prologue path: N(0,1) entries times a
    # per-row power of two in [2^-3, 2^3] (exact in bf16), so row norms spread
    # over about 1.4 .. 91
    x = rng.standard_normal((rows, heads, d), dtype=np.float32)
    e = rscale.integers(-3, 4, size=(rows, heads, 1))
    return (x * np.exp2(e).astype(np.float32)).astype(np.float32)


def make_problem(
    *,
    seed: int,
    B: int,
    T: int | None = None,
    lengths=None,
    nk: int,
    nv: int,
    dk: int = 128,
    dv: int = 128,
    gate_mu: float = 0.0,
    gate_sigma: float = 1.0,
    gate_zero: bool = False,
    h0_std: float = 0.0,
    h0_mask=None,
    pad_qk: int = 0,
    pad_v: int = 0,
    gb_stride: int | None = None,
    qk_raw: bool = False,
    name: str = "",
) -> Problem:
    """Draw one problem.

    Dense when ``lengths`` is None (B sequences of T tokens each); varlen when
    ``lengths`` is given (B = len(lengths), T = their sum, cu_seqlens built
    from them). ``h0_mask[s]`` selects which sequences get a N(0, h0_std)
    state (others start at zero). ``pad_qk``/``pad_v`` widen the row strides of
    q/k and v beyond the packed minimum; ``gb_stride`` sets the row stride of
    g and beta (the packed conv layout uses 2*nv). ``qk_raw`` leaves the q and k
    head rows un-normalised (the input of the fused L2-norm prologue), with a
    per-row power-of-two scale drawn from an eighth child stream.
    """
    ss = np.random.SeedSequence(seed)
    rq, rk, rv, rg, rb, rh, rl = [np.random.Generator(np.random.PCG64(c)) for c in ss.spawn(7)]
    del rl  # lengths are passed in explicitly (see draw_lengths)
    if lengths is None:
        assert T is not None
        cu = None
        rows = B * T
    else:
        lengths = [int(x) for x in lengths]
        assert len(lengths) == B
        cu = np.zeros(B + 1, dtype=np.int32)
        cu[1:] = np.cumsum(lengths)
        rows = int(cu[-1])
        T = rows
    qs = nk * dk + pad_qk
    vs = nv * dv + pad_v
    gs = nv if gb_stride is None else gb_stride
    assert gs >= nv

    q = np.zeros((rows, qs), dtype=np.uint16)
    k = np.zeros((rows, qs), dtype=np.uint16)
    v = np.zeros((rows, vs), dtype=np.uint16)
    if qk_raw:
        rs = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed).spawn(8)[7]))
        qf = _raw_rows(rq, rs, rows, nk, dk)
        kf = _raw_rows(rk, rs, rows, nk, dk)
    else:
        qf = _normalised_rows(rq, rows, nk, dk)
        kf = _normalised_rows(rk, rows, nk, dk)
    q[:, : nk * dk] = f32_to_bf16_bits(qf.reshape(rows, nk * dk))
    k[:, : nk * dk] = f32_to_bf16_bits(kf.reshape(rows, nk * dk))
    v[:, : nv * dv] = f32_to_bf16_bits(rv.standard_normal((rows, nv * dv), dtype=np.float32))

    g = np.zeros((rows, gs), dtype=np.float32)
    beta = np.zeros((rows, gs), dtype=np.float32)
    if gate_zero:
        g[:, :nv] = 0.0
        rg.standard_normal((rows, nv))  # keep the stream position identical
    else:
        x = rg.standard_normal((rows, nv)) * gate_sigma + gate_mu
        g[:, :nv] = (-_softplus(x)).astype(np.float32)
    beta[:, :nv] = (1.0 / (1.0 + np.exp(-rb.standard_normal((rows, nv))))).astype(np.float32)

    h0 = np.zeros((B, nv, dk, dv), dtype=np.float32)
    if h0_std > 0:
        draw = (rh.standard_normal((B, nv, dk, dv), dtype=np.float32) * np.float32(h0_std)).astype(np.float32)
        mask = np.ones(B, dtype=bool) if h0_mask is None else np.asarray(h0_mask, dtype=bool)
        h0[mask] = draw[mask]
    return Problem(B=B, T=T, nk=nk, nv=nv, dk=dk, dv=dv, q=q, k=k, v=v, g=g, beta=beta,
                   h0=h0, cu_seqlens=cu, name=name, meta={"qk_raw": qk_raw})


def draw_lengths(seed: int, n: int, lo: int, hi: int, avoid_multiple: int = 64):
    """n integer lengths uniform in [lo, hi], redrawing multiples of ``avoid_multiple``."""
    ss = np.random.SeedSequence(seed)
    rl = np.random.Generator(np.random.PCG64(ss.spawn(7)[6]))
    out = []
    while len(out) < n:
        x = int(rl.integers(lo, hi + 1))
        if avoid_multiple and x % avoid_multiple == 0:
            continue
        out.append(x)
    return out


# The five workloads (shapes and distributions) the prefill is specified on.
CONFIGS = {
    0: dict(B=1, T=256, nk=1, nv=1, h0_std=0.0),
    1: dict(B=1, T=4096, nk=16, nv=32, h0_std=0.0),
    2: dict(B=4, T=8192, nk=16, nv=32, h0_std=0.02),
    3: dict(B=8, lengths="draw", nk=16, nv=48, h0_std=0.02, h0_mask="odd"),
    4: dict(B=1, T=65536, nk=16, nv=32, h0_std=0.0, gate_mu=-3.0, gate_sigma=0.5),
}

CONFIG_NAMES = {
    0: "B=1 T=256 nk=nv=1 dk=dv=128",
    1: "B=1 T=4096 nk=16 nv=32 dk=dv=128",
    2: "B=4 T=8192 nk=16 nv=32 dk=dv=128 h0~N(0,0.02)",
    3: "varlen 8 seqs len~U[100,16000] nk=16 nv=48 dk=dv=128 state table",
    4: "B=1 T=65536 nk=16 nv=32 dk=dv=128 g=-softplus(N(-3,0.5))",
}


def config_problem(index: int, **overrides) -> Problem:
    """The seeded problem for workload ``index`` (seed 1000 + index)."""
    c = dict(CONFIGS[index])
    c.update(overrides)
    seed = c.pop("seed", 1000 + index)
    if c.get("lengths") == "draw":
        c["lengths"] = draw_lengths(seed, c["B"], 100, 16000)
    if c.get("h0_mask") == "odd":
        c["h0_mask"] = [s % 2 == 1 for s in range(c["B"])]
    p = make_problem(seed=seed, name=CONFIG_NAMES.get(index, f"config{index}"), **c)
    p.meta["config"] = index
    p.meta["state_table"] = index == 3
    return p
