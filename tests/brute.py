"""Scalar brute-force restatement of the block forward, for pinning the oracle on tiny inputs.

Pure Python loops over lists of floats (math.exp, math.sqrt): no NumPy, no shared helpers with
``oracle/``. It takes the separate Q, K and V projection matrices and the un-interleaved gate/up
matrices, so the oracle's fused-weight row orders (all-Q, all-K, all-V; gate j at row 2j, up j at
row 2j + 1) are checked by construction.
"""

import math


def matvec(W, x):
    return [sum(W[o][i] * x[i] for i in range(len(x))) for o in range(len(W))]


def rmsnorm_row(x, eps):
    ms = sum(v * v for v in x) / len(x)
    r = 1.0 / math.sqrt(ms + eps)
    return [v * r for v in x]


def block(x, Wq, Wk, Wv, Wo, Wg, Wu, Wd, mod_rows, cos, sin, heads, d, eps, qk_eps,
          norm1=None, norm2=None, qn=None, kn=None, post_attn=None, post_mlp=None, linear=None):
    """x: list of R rows (lists of H floats). mod_rows[r] = 6 lists of H (shift_a, scale_a, gate_a,
    shift_m, scale_m, gate_m) for row r. cos/sin: R lists of d/2. Returns new rows.
    linear(W, row) replaces the plain W row products when given (one call per weight matrix)."""
    return _block(x, Wq, Wk, Wv, Wo, Wg, Wu, Wd, mod_rows, cos, sin, heads, d, eps, qk_eps,
                  norm1, norm2, qn, kn, post_attn, post_mlp, linear or matvec)


def _block(x, Wq, Wk, Wv, Wo, Wg, Wu, Wd, mod_rows, cos, sin, heads, d, eps, qk_eps,
           norm1, norm2, qn, kn, post_attn, post_mlp, matvec):
    R, H = len(x), len(x[0])
    one = lambda n: [1.0] * n
    n1 = norm1 or one(H)
    n2 = norm2 or one(H)
    qn = qn or one(d)
    kn = kn or one(d)

    def modnorm(row, w, shift, scale):
        y = rmsnorm_row(row, eps)
        return [y[i] * w[i] * (1.0 + scale[i]) + shift[i] for i in range(H)]

    Q, K, V = [], [], []
    for r in range(R):
        sa, ca = mod_rows[r][0], mod_rows[r][1]
        h = modnorm(x[r], n1, sa, ca)
        q, k, v = matvec(Wq, h), matvec(Wk, h), matvec(Wv, h)
        qh, kh, vh = [], [], []
        for n in range(heads):
            for (src, w, dst) in ((q, qn, qh), (k, kn, kh)):
                seg = rmsnorm_row(src[n * d:(n + 1) * d], qk_eps)
                seg = [seg[j] * w[j] for j in range(d)]
                rot = [0.0] * d
                for i in range(d // 2):
                    a, b = seg[2 * i], seg[2 * i + 1]
                    c, s = cos[r][i], sin[r][i]
                    rot[2 * i] = a * c - b * s
                    rot[2 * i + 1] = a * s + b * c
                dst.append(rot)
            vh.append(v[n * d:(n + 1) * d])
        Q.append(qh)
        K.append(kh)
        V.append(vh)

    out = []
    for r in range(R):
        o = []
        for n in range(heads):
            scores = [sum(Q[r][n][j] * K[c][n][j] for j in range(d)) / math.sqrt(d) for c in range(R)]
            m = max(scores)
            e = [math.exp(s - m) for s in scores]
            z = sum(e)
            for j in range(d):
                o.append(sum(e[c] / z * V[c][n][j] for c in range(R)))
        att = matvec(Wo, o)
        if post_attn is not None:
            att = [v * w for v, w in zip(rmsnorm_row(att, eps), post_attn)]
        ga = mod_rows[r][2]
        xr = [x[r][i] + ga[i] * att[i] for i in range(H)]
        sm, cm, gm = mod_rows[r][3], mod_rows[r][4], mod_rows[r][5]
        h2 = modnorm(xr, n2, sm, cm)
        g, u = matvec(Wg, h2), matvec(Wu, h2)
        a = [g[j] / (1.0 + math.exp(-g[j])) * u[j] for j in range(len(g))]
        mlp = matvec(Wd, a)
        if post_mlp is not None:
            mlp = [v * w for v, w in zip(rmsnorm_row(mlp, eps), post_mlp)]
        out.append([xr[i] + gm[i] * mlp[i] for i in range(H)])
    return out


def layernorm_row(x, eps):
    mu = sum(x) / len(x)
    var = sum((v - mu) * (v - mu) for v in x) / len(x)
    r = 1.0 / math.sqrt(var + eps)
    return [(v - mu) * r for v in x]


def parallel_block(x, Wq, Wk, Wv, Wo, Wg, Wu, Wd, mod_rows, cos, sin, heads, d, eps, qk_eps,
                   norm=None, qn=None, kn=None, linear=None, linear2=None, post_attn=None, post_mlp=None):
    """The parallel block: x + gate * (attention + SwiGLU MLP), both branches reading one modulated
    LayerNorm. mod_rows[r] = 3 lists of H (shift, scale, gate) for row r. Returns new rows.
    linear(W, row) replaces the products of Wq, Wk, Wv, Wg and Wu when given; linear2(o, a) replaces
    the sum of the two output products Wo o + Wd a (one linear over the joined input [o | a]).
    post_attn / post_mlp: each branch's output RMS-normed times its weight before the shared gate."""
    if post_attn is not None or post_mlp is not None:
        assert linear2 is None, "post norms need the two output products apart"

        def joint(o, a):
            att, mlp = matvec(Wo, o), matvec(Wd, a)
            if post_attn is not None:
                att = [v * w for v, w in zip(rmsnorm_row(att, eps), post_attn)]
            if post_mlp is not None:
                mlp = [v * w for v, w in zip(rmsnorm_row(mlp, eps), post_mlp)]
            return [u + v for u, v in zip(att, mlp)]
        linear2 = joint
    matvec_ = linear or matvec
    joint = linear2 or (lambda o, a: [u + v for u, v in zip(matvec(Wo, o), matvec(Wd, a))])
    R, H = len(x), len(x[0])
    one = lambda n: [1.0] * n
    w = norm or one(H)
    qn = qn or one(d)
    kn = kn or one(d)
    hs, Q, K, V = [], [], [], []
    for r in range(R):
        shift, scale = mod_rows[r][0], mod_rows[r][1]
        y = layernorm_row(x[r], eps)
        h = [y[i] * w[i] * (1.0 + scale[i]) + shift[i] for i in range(H)]
        hs.append(h)
        q, k, v = matvec_(Wq, h), matvec_(Wk, h), matvec_(Wv, h)
        qh, kh, vh = [], [], []
        for n in range(heads):
            for (src, wt, dst) in ((q, qn, qh), (k, kn, kh)):
                seg = rmsnorm_row(src[n * d:(n + 1) * d], qk_eps)
                seg = [seg[j] * wt[j] for j in range(d)]
                rot = [0.0] * d
                for i in range(d // 2):
                    a, b = seg[2 * i], seg[2 * i + 1]
                    c, s = cos[r][i], sin[r][i]
                    rot[2 * i] = a * c - b * s
                    rot[2 * i + 1] = a * s + b * c
                dst.append(rot)
            vh.append(v[n * d:(n + 1) * d])
        Q.append(qh)
        K.append(kh)
        V.append(vh)
    out = []
    for r in range(R):
        o = []
        for n in range(heads):
            scores = [sum(Q[r][n][j] * K[c][n][j] for j in range(d)) / math.sqrt(d) for c in range(R)]
            m = max(scores)
            e = [math.exp(s - m) for s in scores]
            z = sum(e)
            for j in range(d):
                o.append(sum(e[c] / z * V[c][n][j] for c in range(R)))
        g, u = matvec_(Wg, hs[r]), matvec_(Wu, hs[r])
        a = [g[j] / (1.0 + math.exp(-g[j])) * u[j] for j in range(len(g))]
        both = joint(o, a)
        gate = mod_rows[r][2]
        out.append([x[r][i] + gate[i] * both[i] for i in range(H)])
    return out


def double_block(x, L, Wt, Wi, mod_rows, cos, sin, heads, d, eps, qk_eps, norms_t=None, norms_i=None,
                 linear=None, post_t=None, post_i=None):
    """The sequential block with per-stream weights: rows r < L use Wt = (Wq, Wk, Wv, Wo, Wg, Wu, Wd)
    and norms_t = (norm1, norm2, qn, kn), the others Wi / norms_i; one attention over all rows.
    linear(W, row) replaces the plain W row products when given (one call per weight matrix).
    post_t / post_i: each stream's (post_attn, post_mlp) sandwich weights (None: un-normed)."""
    matvec = linear or globals()["matvec"]
    posts = (post_t or (None, None), post_i or (None, None))

    def post(y, w):
        return y if w is None else [v * c for v, c in zip(rmsnorm_row(y, eps), w)]
    R, H = len(x), len(x[0])
    one = lambda n: [1.0] * n
    nt = norms_t or (None, None, None, None)
    ni = norms_i or (None, None, None, None)
    pick = lambda r: (Wt, nt) if r < L else (Wi, ni)

    def modnorm(row, w, shift, scale):
        y = rmsnorm_row(row, eps)
        w = w or one(H)
        return [y[i] * w[i] * (1.0 + scale[i]) + shift[i] for i in range(H)]

    Q, K, V = [], [], []
    for r in range(R):
        W, nr = pick(r)
        h = modnorm(x[r], nr[0], mod_rows[r][0], mod_rows[r][1])
        q, k, v = matvec(W[0], h), matvec(W[1], h), matvec(W[2], h)
        qn, kn = nr[2] or one(d), nr[3] or one(d)
        qh, kh, vh = [], [], []
        for n in range(heads):
            for (src, wt, dst) in ((q, qn, qh), (k, kn, kh)):
                seg = rmsnorm_row(src[n * d:(n + 1) * d], qk_eps)
                seg = [seg[j] * wt[j] for j in range(d)]
                rot = [0.0] * d
                for i in range(d // 2):
                    a, b = seg[2 * i], seg[2 * i + 1]
                    c, s = cos[r][i], sin[r][i]
                    rot[2 * i] = a * c - b * s
                    rot[2 * i + 1] = a * s + b * c
                dst.append(rot)
            vh.append(v[n * d:(n + 1) * d])
        Q.append(qh)
        K.append(kh)
        V.append(vh)
    out = []
    for r in range(R):
        W, nr = pick(r)
        o = []
        for n in range(heads):
            scores = [sum(Q[r][n][j] * K[c][n][j] for j in range(d)) / math.sqrt(d) for c in range(R)]
            m = max(scores)
            e = [math.exp(s - m) for s in scores]
            z = sum(e)
            for j in range(d):
                o.append(sum(e[c] / z * V[c][n][j] for c in range(R)))
        pw = posts[0] if r < L else posts[1]
        att = post(matvec(W[3], o), pw[0])
        xr = [x[r][i] + mod_rows[r][2][i] * att[i] for i in range(H)]
        h2 = modnorm(xr, nr[1], mod_rows[r][3], mod_rows[r][4])
        g, u = matvec(W[4], h2), matvec(W[5], h2)
        a = [g[j] / (1.0 + math.exp(-g[j])) * u[j] for j in range(len(g))]
        mlp = post(matvec(W[6], a), pw[1])
        out.append([xr[i] + mod_rows[r][5][i] * mlp[i] for i in range(H)])
    return out
