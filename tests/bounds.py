"""Error bounds for comparing the CUDA step with the fp64 oracle.

The contract's tolerances (attention within 4e-3 and context within 2e-2
absolute for 16-bit inputs; 1e-5 / 1e-4 for fp32) are the pass bar of every
parity test. On long rows they cannot fail: with N allowed slots an attention
entry is about 1/N and a context entry about 1/sqrt(N), below the bar. These
bounds are the second check. They follow the arithmetic the kernels do, so a
plausible mistake (a dropped term, a missing slot, a scaled row) exceeds them
at any row length.

Model. The inputs are exact; u is the unit roundoff of the output dtype (2^-24
fp32, 2^-8 bf16, 2^-11 fp16), u32 = 2^-24.

* Scores s_j = scale * sum_d q_d k_jd are summed in fp32 (tensor cores and
  CUDA-core FMAs alike), so |ds_j| <= gamma_{D+4} * S with
  S = max_j scale * sum_d |q_d||k_jd| (the worst-case dot-product bound,
  Higham, "Accuracy and Stability of Numerical Algorithms", section 3.1; the
  extra 4 covers the scale * log2(e) product and the base-2 exponent).
  Subtracting the computed maximum doubles it: eps_s = 2 gamma_{D+4} S.
* An attention entry a_j = exp(s_j - m) / l carries eps_s (its numerator), up
  to eps_s plus the sum's error (its normaliser l), the exp2 error (a few u32
  each), a stored P (fp16 on the tensor-core path) and the output rounding u:
  |a_j - a_ref| <= r_a a_ref + f, with
  r_a = u + u_P + 2 eps_s + lambda sqrt(N) u32 + 16 u32, and f the absolute
  floor of fp16 subnormals (2^-24, one subnormal spacing: a stored fp16 P and a
  16-bit output each round to half of it), 2^-126 for fp32 (flush to zero).
* A context entry c = sum_j a_j V_j: each weight's own score error (eps_s,
  worst case), the fp32 sums over N slots (the probabilistic bound
  lambda sqrt(N) u32 * sum_j a_j |V_j| of Higham and Mary, "A New Approach to
  Probabilistic Rounding Error Analysis", SIAM J. Sci. Comput. 2019), the
  rounding of P to a 16-bit tensor-core operand (u_op, independent per slot:
  by Hoeffding's inequality |sum_j a_j V_j delta_j| <= lambda u_op
  sqrt(sum_j (a_j V_j)^2) except with probability 2 exp(-lambda^2 / 2)), the
  normaliser's relative error delta_l and the output rounding:
  |c - c_ref| <= (u + delta_l) |c_ref| + (eps_s + lambda sqrt(N) u32) A
                 + lambda sqrt(sum_j ((u_op a_j + f/2) V_j)^2) + 2^-126,
  with A = sum_j a_j |V_j| and delta_l = eps_s + lambda sqrt(N) u32 + 16 u32.

lambda = 8: a failure probability below 3e-14 per entry under Hoeffding.
"""
from __future__ import annotations

import numpy as np
import torch

U32 = 2.0 ** -24
UNIT = {torch.float32: 2.0 ** -24, torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}
# P as stored for the attention rows (fp32 scores on the CUDA-core paths of fp32
# inputs, fp16 P on the tensor-core path of 16-bit inputs) and as the operand
# of the P.V product (the input dtype on the tensor cores)
UNIT_P_STORED = {torch.float32: 2.0 ** -24, torch.bfloat16: 2.0 ** -11,
                 torch.float16: 2.0 ** -11}
UNIT_P_OPERAND = {torch.float32: 2.0 ** -24, torch.bfloat16: 2.0 ** -8,
                  torch.float16: 2.0 ** -11}
FLOOR = {torch.float32: 2.0 ** -126, torch.bfloat16: 2.0 ** -24, torch.float16: 2.0 ** -24}
TINY = 2.0 ** -126
LAMBDA = 8.0


def _gamma(n: int) -> float:
    return n * U32 / (1.0 - n * U32)


class RowBounds:
    """Bounds for the query rows of one batch row (see the module docstring).

    r_att [Hq, Q, 1]: relative bound of the attention entries; floor: their
    absolute floor; rel_ctx [Hq, Q, 1] and abs_ctx [Hq, Q, Dv]: the context
    bound rel_ctx |c_ref| + abs_ctx. Rows t >= n get zero bounds: their
    outputs must be exactly zero."""

    def __init__(self, r_att, floor, rel_ctx, abs_ctx):
        self.r_att, self.floor, self.rel_ctx, self.abs_ctx = r_att, floor, rel_ctx, abs_ctx


def row_bounds(q, K, V, L: int, n: int, scale: float, dtype, att_ref) -> RowBounds:
    """q [Hq, Q, D], K [Hk, M, D], V [Hk, M, Dv]: float64 arrays (K and V the
    updated caches); att_ref [Hq, Q, M]: the oracle's attention (float64);
    L, n: the batch row's old length and append count."""
    q, K, V, att_ref = (np.asarray(a, dtype=np.float64) for a in (q, K, V, att_ref))
    Hq, Q, D = q.shape
    Hk, M, Dv = V.shape
    G = Hq // Hk
    u, up, uo, f = UNIT[dtype], UNIT_P_STORED[dtype], UNIT_P_OPERAND[dtype], FLOOR[dtype]
    r_att = np.zeros((Hq, Q, 1))
    rel_ctx = np.zeros((Hq, Q, 1))
    abs_ctx = np.zeros((Hq, Q, Dv))
    nv = min(n, Q)
    if nv <= 0:
        return RowBounds(r_att, f, rel_ctx, abs_ctx)
    gD = _gamma(D + 4)
    Nmax = L + nv
    for k in range(Hk):
        qa = np.abs(q[k * G:(k + 1) * G, :nv]).reshape(G * nv, D)     # rows (h, t)
        S_all = scale * (qa @ np.abs(K[k, :Nmax]).T)                   # [G*nv, Nmax]
        t_of = np.tile(np.arange(nv), G)
        N_of = L + t_of + 1
        allowed = np.arange(Nmax)[None, :] < N_of[:, None]
        S = np.where(allowed, S_all, 0.0).max(1)
        eps_s = 2.0 * gD * S
        sum_err = LAMBDA * np.sqrt(N_of) * U32
        a = att_ref[k * G:(k + 1) * G, :nv, :Nmax].reshape(G * nv, Nmax)
        Vk = V[k, :Nmax]
        A = a @ np.abs(Vk)
        w = np.where(allowed, uo * a + 0.5 * f, 0.0)
        B = np.sqrt((w ** 2) @ (Vk ** 2))
        ra = u + up + 2.0 * eps_s + sum_err + 16.0 * U32
        rc = u + eps_s + sum_err + 16.0 * U32
        ac = (eps_s + sum_err)[:, None] * A + LAMBDA * B + TINY
        r_att[k * G:(k + 1) * G, :nv, 0] = ra.reshape(G, nv)
        rel_ctx[k * G:(k + 1) * G, :nv, 0] = rc.reshape(G, nv)
        abs_ctx[k * G:(k + 1) * G, :nv] = ac.reshape(G, nv, Dv)
    return RowBounds(r_att, f, rel_ctx, abs_ctx)


def attention_ratio(att, att_ref, bnd: RowBounds) -> float:
    """max |att - att_ref| / (r_att |att_ref| + floor); <= 1 passes. Entries
    whose reference is exactly zero must be exactly zero (ratio inf else)."""
    att = np.asarray(att, dtype=np.float64)
    err = np.abs(att - att_ref)
    tol = bnd.r_att * np.abs(att_ref) + np.where(att_ref != 0.0, bnd.floor, 0.0)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(err == 0.0, 0.0, err / tol)
    return float(r.max(initial=0.0))


def context_ratio(ctx, ctx_ref, bnd: RowBounds) -> float:
    """max |ctx - ctx_ref| / (rel_ctx |ctx_ref| + abs_ctx); <= 1 passes."""
    ctx = np.asarray(ctx, dtype=np.float64)
    err = np.abs(ctx - ctx_ref)
    tol = bnd.rel_ctx * np.abs(ctx_ref) + bnd.abs_ctx
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(err == 0.0, 0.0, err / tol)
    return float(r.max(initial=0.0))


def check_rows(att, ctx, att_ref, ctx_ref, bnd: RowBounds, where: str = ""):
    """Assert both ratios <= 1 and that two wrong variants made from the
    oracle's own output (context and attention scaled by 0.9; all-zero
    outputs) exceed the bound wherever the row has valid queries, so the check
    can fail on these rows. Returns the two ratios."""
    ra = attention_ratio(att, att_ref, bnd)
    rc = context_ratio(ctx, ctx_ref, bnd)
    assert ra <= 1.0, f"{where} attention error {ra:.3g} x its bound"
    assert rc <= 1.0, f"{where} context error {rc:.3g} x its bound"
    if np.any(att_ref != 0.0):
        assert attention_ratio(0.9 * att_ref, att_ref, bnd) > 1.0, where
        assert attention_ratio(np.zeros_like(att_ref), att_ref, bnd) > 1.0, where
    if np.any(ctx_ref != 0.0):
        assert context_ratio(0.9 * ctx_ref, ctx_ref, bnd) > 1.0, where
        assert context_ratio(np.zeros_like(ctx_ref), ctx_ref, bnd) > 1.0, where
    return ra, rc


def check_step(inputs, upd_key, upd_value, att, ctx, att_ref, ctx_ref, scale, where=""):
    """check_rows on every batch row of a step. inputs: the StepInputs on the
    CPU; upd_key / upd_value: the updated caches (dtype tensors, bit-exact
    already checked); att / ctx: the GPU results; att_ref / ctx_ref: the
    oracle's (float64). Rows the contract rejects are skipped (their outputs
    are checked to be zero elsewhere). Returns the worst ratios."""
    q = inputs.query.double().numpy()
    K = upd_key.double().numpy()
    V = upd_value.double().numpy()
    mask = inputs.append_mask.to(torch.int64)
    counts = mask.cumprod(1).sum(1).numpy()
    prefix = (mask.sum(1).numpy() == counts)
    lengths = inputs.lengths.numpy()
    att = np.asarray(att, dtype=np.float64)
    ctx = np.asarray(ctx, dtype=np.float64)
    worst = (0.0, 0.0)
    for b in range(q.shape[0]):
        L, n = int(lengths[b]), int(counts[b])
        M = K.shape[2]
        if L < 0 or L + n > M or n == 0 or not prefix[b]:
            continue
        bnd = row_bounds(q[b], K[b], V[b], L, n, scale, inputs.query.dtype, att_ref[b])
        r = check_rows(att[b], ctx[b], att_ref[b], ctx_ref[b], bnd, f"{where} batch row {b}")
        worst = (max(worst[0], r[0]), max(worst[1], r[1]))
    return worst


# ---------------------------------------------------------------- gradients
# |got - ref| <= rtol |ref| + atol (RMS(ref) + T) + floor per entry, with RMS
# over the tensor's nonzero reference entries and T the root of the sum of
# squares of the entry's own terms (grad_terms).
#
# rtol covers the final rounding of a gradient and, on the tensor-core slot
# kernel, the rounding of a and ds to 16-bit operands (2u for bf16, 4u for
# fp16). atol covers the sums of independently rounded terms, whose error is
# relative to the terms' magnitude rather than to the (possibly cancelled)
# entry: by Hoeffding's inequality at most lambda u T, with lambda = 8 as for
# the forward bounds, so atol = 8u (2^-5 bf16, 2^-8 fp16); fp32 keeps 1e-4 for
# its fp32 sums over up to 1e5 slots. The RMS term is the tensor-wide share of
# the errors of the rows' shared fp32 statistics (normaliser, maximum, D).
# The floor is one fp16 subnormal spacing (long-row cache gradients are fp16
# subnormals) or fp32's flush-to-zero threshold.
#
# The entries the step's structure makes zero (exact_zero: invalid query
# rows, new rows nothing appended) must be exactly zero. Any other entry may
# be zero by cancellation (a row with two allowed slots has ds_0 = -ds_1, so
# its query gradient vanishes wherever the two keys agree) and keeps the atol
# term: the fp32 sums leave a residue there.
GRAD_TOL = {torch.bfloat16: (2.0 ** -7, 2.0 ** -5), torch.float16: (2.0 ** -9, 2.0 ** -8),
            torch.float32: (1e-4, 1e-4)}
GRAD_FLOOR = {torch.bfloat16: TINY, torch.float16: 2.0 ** -24, torch.float32: TINY}


def grad_ratio(got, ref, dtype, exact_zero=None, terms=None) -> float:
    """max |got - ref| / (rtol |ref| + atol (RMS(ref) + T) + floor); <= 1 passes.
    exact_zero (boolean, ref's shape, or None): entries that must be zero.
    terms (ref's shape, or None for zero): T, the root of the sum of squares of
    the terms each entry sums (grad_terms)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rtol, atol = GRAD_TOL[dtype]
    nz = ref[ref != 0.0]
    rms = float(np.sqrt(np.mean(nz ** 2))) if nz.size else 0.0
    err = np.abs(got - ref)
    spread = rms if terms is None else rms + np.asarray(terms, dtype=np.float64)
    tol = rtol * np.abs(ref) + atol * spread + GRAD_FLOOR[dtype]
    if exact_zero is not None:
        tol = np.where(exact_zero, 0.0, tol)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(err == 0.0, 0.0, err / tol)
    return float(r.max(initial=0.0))


def grad_terms(query, lengths, append_mask, fwd, d_attention, d_context, scale, sums=False):
    """T per gradient entry: the root of the sum of squares of the terms it
    sums, from the oracle's forward pass fwd (oracle.step: attention rows a
    and updated caches K', V') and the incoming gradients (None: zero). For a
    valid row r of a unit and an allowed slot j, with g_rj = dattention_rj +
    dcontext_r . V'_j, D_r = sum_j a_rj g_rj and ds_rj = a_rj (g_rj - D_r):

      dK'_j: scale sqrt(sum_r (ds_rj q_r)^2)     dV'_j: sqrt(sum_r (a_rj dcontext_r)^2)
      dq_r:  scale sqrt(sum_j (ds_rj K'_j)^2)

    elementwise over the width; a new row's gradient takes its slot's. The
    16-bit rounding of a and ds (independent per term) moves an entry by at
    most lambda u T (Hoeffding), which on a row of few slots, whose terms are
    large next to the tensor's RMS, is the larger part of the error.
    Returns a dict keyed like the gradients (query, new_key, new_value,
    key_cache, value_cache); with sums, also the terms' plain sums (the
    attention-derived part of each gradient) under "sum_" + key."""
    q = np.asarray(query.double().numpy() if torch.is_tensor(query) else query, dtype=np.float64)
    K = fwd["key_cache"].double().numpy()
    V = fwd["value_cache"].double().numpy()
    att = np.asarray(fwd["attention"], dtype=np.float64)
    B, Hq, Q, D = q.shape
    Hk, M, Dv = V.shape[1], V.shape[2], V.shape[3]
    G = Hq // Hk
    da = (np.zeros((B, Hq, Q, M)) if d_attention is None else d_attention.double().numpy())
    dc = (np.zeros((B, Hq, Q, Dv)) if d_context is None else d_context.double().numpy())
    counts = append_mask.to(torch.int64).cumprod(1).sum(1).numpy()
    ln = lengths.numpy()
    shapes = {"query": (B, Hq, Q, D), "new_key": (B, Hk, Q, D), "new_value": (B, Hk, Q, Dv),
              "key_cache": (B, Hk, M, D), "value_cache": (B, Hk, M, Dv)}
    out = {k: np.zeros(v) for k, v in shapes.items()}
    if sums:
        out.update({"sum_" + k: np.zeros(v) for k, v in shapes.items()})
    for b in range(B):
        L, n = int(ln[b]), int(counts[b])
        if fwd["flags"][b] or n == 0:
            continue
        N = L + n
        for kv in range(Hk):
            hs = slice(kv * G, (kv + 1) * G)
            a = att[b, hs, :n, :N].reshape(G * n, N)
            Kp, Vp = K[b, kv, :N], V[b, kv, :N]
            qr = q[b, hs, :n].reshape(G * n, D)
            dcr = dc[b, hs, :n].reshape(G * n, Dv)
            g = da[b, hs, :n, :N].reshape(G * n, N) + dcr @ Vp.T
            ds = a * (g - (a * g).sum(1, keepdims=True))
            Tk = scale * np.sqrt((ds ** 2).T @ (qr ** 2))
            Tv = np.sqrt((a ** 2).T @ (dcr ** 2))
            Tq = scale * np.sqrt((ds ** 2) @ (Kp ** 2))
            out["key_cache"][b, kv, :L] = Tk[:L]
            out["new_key"][b, kv, :n] = Tk[L:N]
            out["value_cache"][b, kv, :L] = Tv[:L]
            out["new_value"][b, kv, :n] = Tv[L:N]
            out["query"][b, hs, :n] = Tq.reshape(G, n, D)
            if sums:
                Sk, Sv, Sq = scale * (ds.T @ qr), a.T @ dcr, scale * (ds @ Kp)
                out["sum_key_cache"][b, kv, :L] = Sk[:L]
                out["sum_new_key"][b, kv, :n] = Sk[L:N]
                out["sum_value_cache"][b, kv, :L] = Sv[:L]
                out["sum_new_value"][b, kv, :n] = Sv[L:N]
                out["sum_query"][b, hs, :n] = Sq.reshape(G, n, D)
    return out
