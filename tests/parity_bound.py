"""Per-element error bounds of the library's GEMV arithmetic, and an emulation of it.

The parity bar of every GEMV test is a normalized error of 2e-3. Beside it the
tests check each output element against a bound derived from the arithmetic
the kernels do, which is far tighter where that arithmetic is exact:

CUDA-core path (vbq_gemv, and every projection of vbq_decode_step):
  * a row's partial sums are integers in units of 2^-F, F = 30 - (e(L1) + e(max|x|)),
    e(v) the exponent with v < 2^e, L1 the largest row sum of |w| rounded up to
    fp32; each (row, group) entry adds round(v) for its real contribution v,
    an error of at most half a unit;
  * 1-bit groups: v = s * sum of 13 table values, each a 5-term fp32 sum of
    +-x * 2^F / 2: fp32 rounding of at most 24 * 2^-24 * |s| * sum|x| / 2;
  * 2-, 4- and 8-bit groups: x is rounded to X = rint(x * 2^s_g), s_g = 14 -
    e(max over the group of |x|), so the dot product is exact in integers but
    off by |s| * sum|q - c| * 2^-(s_g + 1); three fp32 roundings follow;
  * the 64-bit sum is rounded once to fp32.
In the decode step each CTA's F is at least the F of the whole input, and its
64-bit sums carry 32 more bits, so the same bound holds with a small slack.

Tensor-core path (vbq_gemm_smallbatch, B >= 2): each weight and each scaled x
is rounded once to fp16 (relative 2^-11) and the products are summed in fp32.

emulate_gemv follows the CUDA-core arithmetic in numpy (fp32 where the kernel
uses fp32). It is test infrastructure: tests check the emulation against the
oracle within the bound, which pins the bound on the CPU.
"""

from __future__ import annotations

import numpy as np

from oracle import vbq_oracle as O

GROUP = 64
U = 2.0 ** -24


def exp_above(v: np.ndarray) -> np.ndarray:
    """e with |v| < 2^e (frexp's exponent); 0 where v == 0."""
    _, e = np.frexp(np.asarray(v, dtype=np.float64))
    return e.astype(np.int64)


def max_row_l1(codes, bits, scales) -> float:
    """The packer's L1 bound: max over rows of sum |w|, rounded up to the next fp32."""
    W = np.abs(O.dequant(codes, bits, scales).astype(np.float64))
    l1 = float(W.sum(axis=1).max()) if W.size else 0.0
    return float(np.nextafter(np.float32(l1), np.float32(3e38)))


def fixed_exponent(l1: float, maxx: float) -> int:
    if not (maxx > 0.0) or not (l1 > 0.0):
        return 0
    return int(30 - (exp_above(np.float32(l1)) + exp_above(np.float32(maxx))))


def group_shift(x: np.ndarray) -> np.ndarray:
    """s_g per group of 64: 14 - e(max|x_g|), 0 for an all-zero group."""
    m = np.abs(x).reshape(-1, GROUP).max(axis=1)
    return np.where(m > 0.0, 14 - exp_above(m), 0)


def cuda_core_bound(codes, bits, scales, x_bits, F: int, slack_units: float = 0.0) -> np.ndarray:
    """Bound on |y - y_exact| per row for the CUDA-core arithmetic with unit 2^-F."""
    n, k = codes.shape
    g = k // GROUP
    x = O.bf16_bits_to_f64(x_bits)
    ax = np.abs(x).reshape(g, GROUP)
    s = np.abs(O.f16_bits_to_f64(scales))                       # [n, g]
    cq = np.abs(O.dequant(codes, bits, np.full_like(scales, 0x3C00)).astype(np.float64)).reshape(n, g, GROUP)
    unit = 2.0 ** -F
    sumx = ax.sum(axis=1)                                       # [g]
    sg = group_shift(x)                                         # [g]
    one = (bits == 1)
    b1 = 24.0 * U * s * 0.5 * sumx[None, :]
    qx = (cq * ax[None]).sum(axis=2)                            # sum |q - c| |x| per entry
    q1 = cq.sum(axis=2)                                         # sum |q - c| per entry
    bdp = s * q1 * np.ldexp(0.5, -sg)[None, :] + 4.0 * U * s * (qx + q1 * np.ldexp(0.5, -sg)[None, :])
    per_entry = np.where(one, b1, bdp) + (0.5 + slack_units) * unit
    total = per_entry.sum(axis=1)
    W = O.dequant(codes, bits, scales).astype(np.float64)
    mag = np.abs(W) @ np.abs(x)
    return total + 2.0 * U * (mag + total)


def gemv_bound(codes, bits, scales, x_bits) -> np.ndarray:
    """The bound for vbq_gemv (F from the matrix's L1 bound and max|x|)."""
    x = O.bf16_bits_to_f64(x_bits)
    F = fixed_exponent(max_row_l1(codes, bits, scales), float(np.abs(x).max()) if x.size else 0.0)
    return cuda_core_bound(codes, bits, scales, x_bits, F)


def tc_bound(codes, bits, scales, X_bits) -> np.ndarray:
    """Bound [B, N] for the tensor-core path: fp16 rounding of w and of x * 2^p, fp32 sums."""
    X = O.bf16_bits_to_f64(X_bits)
    W = np.abs(O.dequant(codes, bits, scales).astype(np.float64))
    k = codes.shape[1]
    mag = np.abs(X) @ W.T                                       # [B, N]
    rel = 2.0 * 2.0 ** -11 + 2.0 ** -22 + (k / 16.0 + 4.0) * 2.0 ** -23
    # fp16 subnormals: absolute error 2^-25 for a weight, 2^-25 / 2^p for an x (max|x| 2^p in [2^13, 2^14))
    mx = np.abs(X).max(axis=1)
    p = np.where(mx > 0.0, 14 - exp_above(mx), 0)
    sub = 2.0 ** -25 * (np.abs(X).sum(axis=1)[:, None] + W.sum(axis=1)[None, :] * np.ldexp(1.0, -p)[:, None])
    return rel * mag + 2.0 * sub + 1e-300


def check_within(y, y_ref, bound) -> float:
    """Largest |y - y_ref| / bound; asserts it is at most 1."""
    d = np.abs(np.asarray(y, np.float64) - np.asarray(y_ref, np.float64))
    r = d / np.maximum(bound, 1e-300)
    worst = float(r.max()) if r.size else 0.0
    assert worst <= 1.0, (worst, np.unravel_index(int(np.argmax(r)), r.shape))
    return worst


# ---- emulation of the CUDA-core arithmetic ----

def _f32(v):
    return np.float32(v)


def emulate_gemv(codes, bits, scales, x_bits) -> np.ndarray:
    """The CUDA-core GEMV's arithmetic, entry by entry, in numpy (fp32 where the kernel is fp32)."""
    n, k = codes.shape
    g = k // GROUP
    x = O.bf16_bits_to_f64(x_bits).astype(np.float32)
    F = fixed_exponent(max_row_l1(codes, bits, scales), float(np.abs(x).max()) if x.size else 0.0)
    xp = (x.astype(np.float64) * 2.0 ** F).astype(np.float32)   # exact while in range
    sg = group_shift(x.astype(np.float64))
    s16 = O.f16_bits_to_f64(scales).astype(np.float32)
    acc = np.zeros(n, dtype=np.int64)
    for j in range(g):
        xs = xp[j * GROUP:(j + 1) * GROUP]
        xe = np.concatenate([xs, np.zeros(6, np.float32)])
        X = np.rint(x[j * GROUP:(j + 1) * GROUP].astype(np.float64) * 2.0 ** int(sg[j])).astype(np.int64)
        u = np.float32(2.0 ** (F - int(sg[j]) - 1))
        for r in range(n):
            b = int(bits[r, j])
            q = codes[r, j * GROUP:(j + 1) * GROUP].astype(np.int64)
            if b == 1:
                a = [np.float32(0.0)] * 4
                for kk in range(13):
                    t = np.float32(0.0)
                    for i in range(5):
                        m = 5 * kk + i
                        qm = int(q[m]) if m < GROUP else 0
                        t = _f32(t + _f32((0.5 if qm else -0.5) * xe[m]))
                    a[kk & 3] = _f32(a[kk & 3] + t)
                v = _f32(s16[r, j] * _f32(_f32(a[0] + a[1]) + _f32(a[2] + a[3])))
            else:
                t2 = 2 * int((q * X).sum()) - ((1 << b) - 1) * int(X.sum())
                v = _f32(s16[r, j] * _f32(_f32(t2) * u))
            acc[r] += int(np.rint(np.float64(v)))
    return np.array([np.float32(np.float32(a) * np.float32(2.0 ** -F)) if abs(F) < 100 else
                     np.float32(np.ldexp(np.float64(np.float32(a)), -F)) for a in acc], dtype=np.float32)


# ---- decode attention ----

def attention_bound(q_bits, k_bits, v_bits, T, p):
    """Per-element bound for fp32 scores (d-term sums), expf, the running sums over
    sub-chunks of 64 positions (a rescale per sub-chunk) and the merge of at most
    64 spans: twice the largest score error, plus the rounding of the weighted
    sums, times sum_j p_j |v_j|."""
    q = O.bf16_bits_to_f64(q_bits)
    K = O.bf16_bits_to_f64(k_bits)[:, :T, :]
    Vv = np.abs(O.bf16_bits_to_f64(v_bits)[:, :T, :])
    H, d = q.shape
    group = H // K.shape[0]
    steps = (T + 63) // 64 + 64
    out = np.zeros((H, d))
    for h in range(H):
        g = h // group
        ds = (d + 2) * 2.0 ** -24 * (np.abs(K[g]) @ np.abs(q[h])) / np.sqrt(d)
        rel = 4.0 * ds.max() + (steps + 140) * 2.0 ** -22
        out[h] = rel * (p[h] @ Vv[g]) + 1e-30
    return out


def emulate_attention(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray, T: int, nparts: int,
                      sub: int = 64, drop_last: bool = False, scale_by_d: bool = False) -> np.ndarray:
    """The split-KV decode attention's arithmetic in numpy fp32: fp32 scores times an fp32 1/sqrt(d);
    per span of whole 64-position sub-chunks a running max, exp(s - m), a rescale by exp(m_old - m) of
    the running sum and of the p-weighted sums of v; then the spans merged with weights exp(m_c - M)
    and one division. The dot products and sums run in numpy's order, not the kernel's, which the
    bound allows. drop_last and scale_by_d plant mistakes (the last position left out; 1/d for
    1/sqrt(d)) for the self-test of the bound. Returns [H, d] fp64 of fp32 values."""
    f32 = np.float32
    q = O.bf16_bits_to_f64(q_bits).astype(f32)
    K = O.bf16_bits_to_f64(k_bits)[:, :T, :].astype(f32)
    Vv = O.bf16_bits_to_f64(v_bits)[:, :T, :].astype(f32)
    H, d = q.shape
    group = H // K.shape[0]
    scale = f32(1.0) / (f32(d) if scale_by_d else np.sqrt(f32(d)))
    Tn = T - 1 if drop_last else T
    nsub = (Tn + sub - 1) // sub
    span_sub = (nsub + nparts - 1) // nparts
    nparts = (nsub + span_sub - 1) // span_sub
    out = np.zeros((H, d), f32)
    with np.errstate(over="ignore", under="ignore"):
        for h in range(H):
            g = h // group
            S = (K[g, :Tn] @ q[h]).astype(f32) * scale
            ms, ls, accs = [], [], []
            for c in range(nparts):
                p0, p1 = c * span_sub * sub, min(Tn, (c + 1) * span_sub * sub)
                m, l, acc = f32(-np.inf), f32(0.0), np.zeros(d, f32)
                for j0 in range(p0, p1, sub):
                    s = S[j0:min(p1, j0 + sub)]
                    mn = max(m, s.max())
                    p = np.exp(s - mn).astype(f32)
                    alpha = np.exp(f32(m - mn)).astype(f32)
                    l = f32(l * alpha + p.sum(dtype=f32))
                    acc = (acc * alpha + p @ Vv[g, j0:j0 + p.size]).astype(f32)
                    m = mn
                ms.append(m)
                ls.append(l)
                accs.append(acc)
            if nparts == 1:
                out[h] = accs[0] * (f32(1.0) / ls[0])
                continue
            M = max(ms)
            w = np.exp(np.array(ms, f32) - M).astype(f32)
            L = f32((w * np.array(ls, f32)).sum(dtype=f32))
            out[h] = (w @ np.array(accs, f32)).astype(f32) / L
    return out.astype(np.float64)


def fakequant_tolerances(W, tau: float, G, Q=None):
    """Per-element tolerances of vbq_fakequant_forward and vbq_fakequant_backward against the fp64
    oracle. Forward: 2e-6 * sum_b |Q_b| / min(tau, 1), for the fp32 log, exp and division of the
    mixture weights (their error grows as tau shrinks) and four fp32 products. dalpha: (70 * 2^-24 +
    2e-6 / min(tau, 1)) * 4 * max_b D'_b / tau per group, D'_b = sum over the group of |G| |Q_b|, for
    the fp32 sums of 64 products and the fp32 weights. Q: the oracle's levels, if already computed."""
    from oracle import fakequant_oracle as F
    if Q is None:
        Q = F.levels(W).astype(np.float64)
    n, k = np.asarray(W).shape
    tol = 2e-6 * np.abs(Q).sum(axis=0) / min(tau, 1.0) + 1e-30
    Dabs = (np.abs(np.asarray(G, np.float64))[None] * np.abs(Q)).reshape(4, n, k // 64, 64).sum(axis=3)
    scale = np.moveaxis(Dabs, 0, -1).max(axis=-1, keepdims=True) / tau
    tol_a = (70 * 2.0 ** -24 + 2e-6 / min(tau, 1.0)) * 4 * scale + 1e-30
    return tol, tol_a


def _fma32(a, b, c):
    """fp32 fma: the fp64 product of two fp32 values is exact; one rounding of the fp64 sum to fp32
    (a double rounding, at most an ulp of fp32 off a true fma, which the tolerances absorb)."""
    return (np.asarray(a, np.float64) * np.asarray(b, np.float64) + np.asarray(c, np.float64)).astype(np.float32)


def emulate_fakequant(W, alpha, u, tau: float, G, tau_multiplies: bool = False, offset_half_range: bool = False,
                      D_without_G: bool = False):
    """The fake-quantization kernels' arithmetic in numpy fp32, with their order: mixture weights from
    fp32 log, exp and a 4-lane butterfly; levels rint(w r_b + c_b) with r_b = c_b / max|w|, each op
    rounded once; the forward an fma chain over b; D_b as 8 lanes of 8-term fma chains (weights 4j..4j+3
    and 32+4j..32+4j+3 of lane j) and a 3-step butterfly; dalpha = (pi_b / tau) (D_b - sum pi D). The
    keyword flags plant mistakes for the self-test. Returns (W_mix [N, K], dalpha [N, K/64, 4]) in fp64."""
    f32 = np.float32
    W = np.asarray(W, f32)
    n, k = W.shape
    g = k // 64
    Wg = W.reshape(n, g, 64)
    inv_tau = f32(tau) if tau_multiplies else f32(1.0) / f32(tau)
    z = ((np.asarray(alpha, f32) - np.log(-np.log(np.asarray(u, f32)))) * inv_tau).astype(f32)  # [n, g, 4]
    m = np.maximum(np.maximum(z[..., 0], z[..., 1]), np.maximum(z[..., 2], z[..., 3]))[..., None]
    e = np.exp((z - m).astype(f32)).astype(f32)
    t = ((e[..., 0] + e[..., 1]).astype(f32) + (e[..., 2] + e[..., 3]).astype(f32)).astype(f32)[..., None]
    pi = (e / t).astype(f32)
    mx = np.abs(Wg).max(axis=2)  # [n, g]
    Q = np.zeros((4, n, g, 64), f32)
    with np.errstate(divide="ignore", invalid="ignore"):
        for i, b in enumerate((1, 2, 4, 8)):
            qmax = f32((1 << b) - 1)
            c = f32(1 << (b - 1)) if offset_half_range else f32(0.5) * qmax
            s = np.where(mx > 0, mx / c, f32(0)).astype(f32)[..., None]
            r = np.where(mx > 0, c / mx, f32(0)).astype(f32)[..., None]
            q = np.clip(np.rint(((Wg * r).astype(f32) + c).astype(f32)), f32(0), qmax)
            Q[i] = (s * (q - c).astype(f32)).astype(f32)
    out = np.zeros((n, g, 64), f32)
    for i in range(4):
        out = _fma32(pi[..., i][..., None], Q[i], out)
    Gg = np.asarray(G, f32).reshape(n, g, 64)
    lanes = np.array([[4 * j + t for t in range(4)] + [32 + 4 * j + t for t in range(4)] for j in range(8)])
    D = np.zeros((n, g, 4), f32)
    for i in range(4):
        prod_g = np.ones_like(Gg) if D_without_G else Gg
        acc = np.zeros((n, g, 8), f32)
        for t in range(8):
            idx = lanes[:, t]
            acc = _fma32(prod_g[..., idx], Q[i][..., idx], acc)
        for dlt in (4, 2, 1):
            acc = (acc + acc[..., np.arange(8) ^ dlt]).astype(f32)
        D[..., i] = acc[..., 0]
    mean = np.zeros((n, g), f32)
    for i in range(4):
        mean = _fma32(pi[..., i], D[..., i], mean)
    da = ((pi * inv_tau).astype(f32) * (D - mean[..., None]).astype(f32)).astype(f32)
    return out.reshape(n, k).astype(np.float64), da.astype(np.float64)
