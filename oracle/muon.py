"""The Muon optimizer step, oracle version (test infrastructure).

Follows the step as the pages describe it:

* "Support Muon in BF16_Optimizer with FP32 gradient accumulation", PR
  description: BF16 micro-batch gradients are accumulated in FP32; Muon runs
  on the original (full) matrices after reduction; only each rank's owned
  intersection of the update is copied back; momentum is FP32 and
  partitioned like the master weights; alignment padding is excluded;
  auxiliary (non-Muon) groups keep their own path.
* "Run Muon once per optimizer step under ZeRO-3, not once per micro-batch",
  "The change": at the step, after the overflow check and before the
  gradient norm, Muon runs once on the accumulated gradient; the gradient
  norm is taken over the Muon updates; a step the loss scaler discards
  leaves the momentum untouched.  Review thread: per-head Muon splits a
  tagged parameter (``muon_num_heads``) into head blocks; untagged
  parameters stay whole.

Readings where the pages are silent:

* momentum m <- beta*m + g in float32 (beta*m rounded, then + g rounded);
* gradient scale: each micro-batch adds scale*g, scale = 1/gas by default;
* per-head: rows split into num_heads contiguous blocks of rows/num_heads,
  each block normalised and orthogonalised on its own; num_heads <= 1 means
  the whole matrix;
* update u = NS(m) (no Nesterov term, no weight decay, no shape factor);
* overflow: any non-finite accumulated gradient element of any parameter
  (padding excluded) skips the step and nothing is written;
* global norm = sqrt(sum over Muon params of ||u||^2 + sum over aux params
  of ||g||^2); coef = min(1, clip / (norm + 1e-6)), clip <= 0 disables;
* write-back: Muon params get accum = coef*u and master -= lr*coef*u;
  aux params get accum = coef*g and their master is left alone (the
  auxiliary optimizer is the caller's).
"""
import numpy as np

from . import newton_schulz as ns

CLIP_EPS = 1e-6


def accumulate(accum, grad, scale, overwrite=False):
    """One micro-batch: accum + scale*grad in float32 (the product is
    rounded to float32 before the sum); overwrite gives scale*grad."""
    sg = np.float32(scale) * np.asarray(grad, np.float32)
    return sg if overwrite else np.asarray(accum, np.float32) + sg


def momentum_update(m, g, beta):
    """m <- beta*m + g in float32 (the product rounded, then the sum)."""
    return np.float32(beta) * np.asarray(m, np.float32) + np.asarray(g, np.float32)


def muon_update(g, m, beta, method="gram", steps=ns.DEFAULT_STEPS, num_heads=0,
                mode="exact"):
    """Momentum update then per-block Newton-Schulz of one Muon matrix.

    Returns (new momentum (float32), update u in the matrix's shape)."""
    m_new = momentum_update(m, g, beta)
    rows = m_new.shape[0]
    h = num_heads if num_heads and num_heads > 1 else 1
    if rows % h:
        raise ValueError("rows must be a multiple of num_heads")
    br = rows // h
    blocks = [ns.newton_schulz(m_new[i * br:(i + 1) * br], method, steps, mode)
              for i in range(h)]
    return m_new, np.vstack(blocks)


def scale_grad(g, grad_scale):
    """g * grad_scale in float32 (a loss scale is undone by passing its
    reciprocal); grad_scale == 1 leaves the gradient as it is."""
    g = np.asarray(g, np.float32)
    return g if grad_scale == 1.0 else np.float32(grad_scale) * g


def adam_update(g, exp_avg, exp_avg_sq, w, lr, beta1, beta2, eps, step):
    """Textbook Adam (Kingma & Ba, 2015) for the auxiliary groups, in float32
    and in this operation order: exp_avg = b1*m + (1-b1)*g;
    exp_avg_sq = b2*v + ((1-b2)*g)*g; denom = sqrt(v)/sqrt(1-b2^t) + eps;
    w = w + (-(lr/(1-b1^t))) * (exp_avg/denom).  The pages keep the
    auxiliary groups on their own Adam path ("Support Muon in BF16_Optimizer
    with FP32 gradient accumulation", PR description); fusing it is this
    library's option."""
    f = np.float32
    g = np.asarray(g, f)
    m = f(beta1) * np.asarray(exp_avg, f) + f(1.0 - beta1) * g
    v = f(beta2) * np.asarray(exp_avg_sq, f) + (f(1.0 - beta2) * g) * g
    bc1 = 1.0 - beta1 ** step
    bc2 = 1.0 - beta2 ** step
    denom = np.sqrt(v) / f(np.sqrt(bc2)) + f(eps)
    w_new = np.asarray(w, f) + f(-(lr / bc1)) * (m / denom)
    return m, v, w_new


def write_back(u, w, post, lr, mode, use_muon):
    """The write-back of one parameter (or any slice of it, element by
    element): v = post * u and, for a Muon parameter, w - lr * v.  exact
    mode keeps a Muon update in float64 until both results are rounded to
    float32 once; otherwise every operation is float32.  An auxiliary
    parameter's master is returned unchanged.  Returns (v, new w)."""
    w = np.asarray(w, np.float32)
    if mode == "exact" and use_muon:
        v64 = post * np.asarray(u, np.float64)
        return v64.astype(np.float32), (w.astype(np.float64) - lr * v64).astype(np.float32)
    v = np.asarray(u, np.float32) if post == 1.0 else np.float32(post) * np.asarray(u, np.float32)
    return v, (w - np.float32(lr) * v if use_muon else w)


def muon_step_full(mats, beta, lr, method="gram", steps=ns.DEFAULT_STEPS, clip=0.0,
                   mode="exact", clip_mode="update", grad_scale=1.0, adam=None):
    """One optimizer step on full matrices (no partition tables).

    mats: list of dicts with keys g (accumulated gradient), m (momentum),
    w (master), use_muon, num_heads, and for auxiliary parameters when
    `adam` is given exp_avg / exp_avg_sq.  Returns a dict with per-parameter
    lists 'update', 'momentum', 'master' (and 'exp_avg', 'exp_avg_sq') and
    scalars 'norm', 'coef', 'applied', 'ns_calls'.

    clip_mode "update" (default): the global norm is taken over the Muon
    updates and the auxiliary gradients, then every update is scaled ("Run
    Muon once per optimizer step under ZeRO-3 ...", "The change").
    clip_mode "grad": the global norm is taken over the gradients and the
    gradients are clipped before Muon runs ("Support Muon in BF16_Optimizer
    with FP32 gradient accumulation", PR description: Muon updates are
    computed after gradient reduction and global clipping).
    grad_scale multiplies the accumulated gradient first, so a loss scale is
    undone before any norm is taken ("Fix Muon optimizer under ZeRO CPU
    offload and bound gather buffers", loss-scaling commit: the clipping
    norm must not see the loss scale).
    adam: dict(lr, beta1, beta2, eps, step) applies adam_update to the
    auxiliary parameters with their clipped gradient."""
    calls0 = ns.NS_CALLS[0]
    gs = [scale_grad(d["g"], grad_scale) for d in mats]
    if any(not np.all(np.isfinite(g)) for g in gs):
        out = {"applied": 0, "norm": 0.0, "coef": 0.0, "ns_calls": 0,
               "update": [np.asarray(d["g"], np.float32) for d in mats],
               "momentum": [np.asarray(d["m"], np.float32) for d in mats],
               "master": [np.asarray(d["w"], np.float32) for d in mats]}
        if adam is not None:
            out["exp_avg"] = [d.get("exp_avg") for d in mats]
            out["exp_avg_sq"] = [d.get("exp_avg_sq") for d in mats]
        return out

    def coef_of(sq):
        norm = float(np.sqrt(sq))
        return norm, (min(1.0, clip / (norm + CLIP_EPS)) if clip > 0 else 1.0)

    def sumsq(arrs):
        sq = 0.0
        for x in arrs:
            x64 = np.asarray(x, np.float64)
            sq += float(np.sum(x64 * x64))
        return sq

    pre = clip_mode == "grad"
    if clip_mode not in ("update", "grad"):
        raise ValueError(clip_mode)
    if pre:
        norm, coef = coef_of(sumsq(gs))
        gin = [g if coef == 1.0 else np.float32(coef) * g for g in gs]
    else:
        gin = gs
    us, moms = [], []
    for d, g in zip(mats, gin):
        if d["use_muon"]:
            m_new, u = muon_update(g, d["m"], beta, method, steps, d.get("num_heads", 0), mode)
        else:
            m_new, u = np.asarray(d["m"], np.float32), g
        moms.append(m_new)
        us.append(u)
    if not pre:
        norm, coef = coef_of(sumsq(us))
    post = 1.0 if pre else coef

    updates, masters, ea, eas = [], [], [], []
    for d, u in zip(mats, us):
        v, w_new = write_back(u, d["w"], post, lr, mode, d["use_muon"])
        if adam is not None and not d["use_muon"]:
            m1, v2, w_new = adam_update(v, d["exp_avg"], d["exp_avg_sq"],
                                        np.asarray(d["w"], np.float32), **adam)
            ea.append(m1)
            eas.append(v2)
        else:
            ea.append(d.get("exp_avg"))
            eas.append(d.get("exp_avg_sq"))
        updates.append(v)
        masters.append(w_new)
    out = {"applied": 1, "norm": norm, "coef": coef,
           "ns_calls": ns.NS_CALLS[0] - calls0,
           "update": updates, "momentum": moms, "master": masters}
    if adam is not None:
        out["exp_avg"] = ea
        out["exp_avg_sq"] = eas
    return out


# ------------------------------------------------ flat, partitioned buffers

def _owned_pieces(params, parts, k):
    """(storage_begin, param_begin, length) for every partition intersecting
    parameter k: the rank-owned intersections of one matrix."""
    off = int(params["offset"][k])
    n = int(params["rows"][k]) * int(params["cols"][k])
    pieces = []
    for q in parts:
        lo = max(off, int(q["flat_begin"]))
        hi = min(off + n, int(q["flat_end"]))
        if lo < hi:
            pieces.append((int(q["storage_offset"]) + lo - int(q["flat_begin"]), lo - off, hi - lo))
    if sum(p[2] for p in pieces) != n:
        raise ValueError(f"parameter {k} is not covered exactly once by the partitions")
    return pieces


def gather_matrix(buf, params, parts, k):
    """Rebuild parameter k's full matrix from the partitioned buffer."""
    rows, cols = int(params["rows"][k]), int(params["cols"][k])
    out = np.empty(rows * cols, dtype=buf.dtype)
    for s, p, n in _owned_pieces(params, parts, k):
        out[p:p + n] = buf[s:s + n]
    return out.reshape(rows, cols)


def scatter_matrix(buf, params, parts, k, mat):
    """Copy each partition's owned intersection of mat back into buf."""
    flat = np.asarray(mat, dtype=buf.dtype).reshape(-1)
    for s, p, n in _owned_pieces(params, parts, k):
        buf[s:s + n] = flat[p:p + n]


def muon_step_flat(accum, momentum, master, params, parts, beta, lr, method="gram",
                   steps=ns.DEFAULT_STEPS, clip=0.0, mode="exact", clip_mode="update",
                   grad_scale=1.0, adam=None, exp_avg=None, exp_avg_sq=None):
    """The step on flat, rank-partitioned storage buffers.

    Reconstructs each parameter from its partitions, runs
    :func:`muon_step_full`, then writes every partition's owned intersection
    of the results back.  Elements no parameter covers (alignment padding,
    gaps between partitions) are never read or written.  Returns new copies
    of (accum, momentum, master) and the result dict; with `adam`, the
    updated exp_avg / exp_avg_sq storage buffers are in the result dict."""
    mats = []
    for k in range(len(params)):
        d = {"g": gather_matrix(accum, params, parts, k),
             "m": gather_matrix(momentum, params, parts, k),
             "w": gather_matrix(master, params, parts, k),
             "use_muon": bool(params["use_muon"][k]),
             "num_heads": int(params["num_heads"][k])}
        if adam is not None and not d["use_muon"]:
            d["exp_avg"] = gather_matrix(exp_avg, params, parts, k)
            d["exp_avg_sq"] = gather_matrix(exp_avg_sq, params, parts, k)
        mats.append(d)
    res = muon_step_full(mats, beta, lr, method, steps, clip, mode, clip_mode, grad_scale, adam)
    acc2, mom2, mst2 = accum.copy(), momentum.copy(), master.copy()
    if adam is not None:
        res["exp_avg_buf"], res["exp_avg_sq_buf"] = exp_avg.copy(), exp_avg_sq.copy()
    if res["applied"]:
        for k in range(len(params)):
            scatter_matrix(acc2, params, parts, k, res["update"][k])
            if mats[k]["use_muon"]:
                scatter_matrix(mom2, params, parts, k, res["momentum"][k])
                scatter_matrix(mst2, params, parts, k, res["master"][k])
            elif adam is not None:
                scatter_matrix(mst2, params, parts, k, res["master"][k])
                scatter_matrix(res["exp_avg_buf"], params, parts, k, res["exp_avg"][k])
                scatter_matrix(res["exp_avg_sq_buf"], params, parts, k, res["exp_avg_sq"][k])
    return acc2, mom2, mst2, res
