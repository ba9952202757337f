"""A validity check of one row of the draft-tree rejection sampler's output,
used where the exact fp64 result and an fp32 kernel may legitimately differ
(a decision within 1e-6 of its threshold).  Plain numpy, independent of the
oracle and of the CUDA library."""
import numpy as np


BAND = 1e-6  # near-boundary band of the sampler (normalised units)


def tree_walk_valid(parent, s, b, k, path, toks):
    """Walk row b of the tree sampler along the GPU's own path in fp64 and check
    every decision it took.  The first child of a node is the fp32 test u*Q <= P
    (bit-exact, no band); a later child's test must agree with
    u*Q(x)*Z <= R(x) unless |u*Q(x)*Z - R(x)| / Z < 1e-6 (the band in which
    fp32 and fp64 residuals may decide differently); after an in-band
    disagreement the walk follows the GPU's decision.  The final token (the
    draw from the residual, or the bonus at a leaf) must have a normalised CDF
    interval that reaches within 1e-6 of u.  Returns (valid, in_band), in_band
    when some decision the GPU took differs from the exact one within the band."""
    P = s.p[b].double().numpy()
    Q = s.q[b].double().numpy()
    tok = s.tokens[b].numpy()
    ua = s.u_accept[b].numpy()
    us = float(s.u_sample[b])
    n = len(parent)
    kids = [[c for c in range(n) if parent[c] == i] for i in range(n)]
    qrow, r = [], 0
    for i in range(n):
        qrow.append(r if kids[i] else -1)
        r += 1 if kids[i] else 0

    def window_ok(R, t):
        if not (0 <= t < R.shape[0]):
            return False
        c = np.cumsum(R)
        if not c[-1] > 0:
            return False
        c = c / c[-1]
        lo = c[t - 1] if t > 0 else 0.0
        return lo - BAND <= us <= c[t] + BAND

    if path[0] != 0:
        return False, False
    node, depth, in_band = 0, 0, False
    while True:
        if not kids[node]:  # a leaf: the bonus comes from its target row
            return depth == k and window_ok(P[node], int(toks[k])), in_band
        nxt = int(path[depth + 1]) if depth < k else -1
        if nxt >= 0 and nxt not in kids[node]:
            return False, in_band
        R, Z = P[node].copy(), 1.0
        Qn = Q[qrow[node]]
        accepted = -1
        for i, c in enumerate(kids[node]):
            x = int(tok[c])
            if i == 0:
                exact = bool(np.float32(ua[c]) * np.float32(Qn[x]) <= np.float32(P[node][x]))
                near = False
            else:
                lhs = float(ua[c]) * Qn[x] * Z
                exact = lhs <= R[x]
                near = Z > 0 and abs(lhs - R[x]) / Z < BAND
            took = nxt == c
            if took != exact:
                if not near:
                    return False, in_band
                in_band = True
            if took:
                accepted = c
                break
            R = np.maximum(R - Z * Qn, 0.0)
            Z = float(R.sum())
        if accepted < 0:
            if nxt >= 0:
                return False, in_band
            t = int(toks[depth])
            if depth != k:
                return False, in_band
            # an empty residual draws from the target row; a residual whose
            # mass is within the band of zero may be empty on either side
            ok = (Z > 0 and window_ok(R, t)) or (Z < BAND and window_ok(P[node], t))
            return ok, in_band
        if int(toks[depth]) != int(tok[accepted]):
            return False, in_band
        depth += 1
        node = accepted
