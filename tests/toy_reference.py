"""A second, independent statement of the tiny decoder, for pinning the oracle.

Pure Python floats on the [out][in] matrices that "The forward pass end to
end" ("The code") draws, written from that page's description of a forward
step: embed, then per layer RMSNorm -> q/k/v -> interleaved RoPE on q and k ->
append K/V -> grouped-query attention over every cached position -> output
projection + residual -> RMSNorm -> SwiGLU -> down projection + residual, then
the final RMSNorm and the output head.  It shares nothing with oracle.c (other
matrix orientation, separate q/k/v and gate/up matrices, lists not arrays),
so agreement between the two pins layout and composition mistakes in either.
"""
import math


def _apply(M, v):
    """M is [out][in]; returns M v."""
    out = []
    for row in M:
        acc = 0.0
        for a, b in zip(row, v):
            acc += a * b
        out.append(acc)
    return out


def _rms_normalise(v, w, eps):
    mean_sq = sum(e * e for e in v) / len(v)
    inv = 1.0 / math.sqrt(mean_sq + eps)
    return [e * inv * g for e, g in zip(v, w)]


def _rotate_pairs(v, n_heads, hd, pos, base):
    """Interleaved: element pairs (2p, 2p+1) of each head turn by pos * base^(-2p/hd)."""
    r = list(v)
    for head in range(n_heads):
        o = head * hd
        for p in range(hd // 2):
            ang = pos * base ** (-(2.0 * p) / hd)
            c, s = math.cos(ang), math.sin(ang)
            x0, x1 = v[o + 2 * p], v[o + 2 * p + 1]
            r[o + 2 * p] = x0 * c - x1 * s
            r[o + 2 * p + 1] = x0 * s + x1 * c
    return r


class ToyDecoder:
    def __init__(self, cfg, W):
        self.cfg, self.W = cfg, W
        self.keys = [[] for _ in range(cfg["n_layer"])]
        self.vals = [[] for _ in range(cfg["n_layer"])]

    def logits(self, token, pos):
        cfg, W = self.cfg, self.W
        hd, nq, nkv = cfg["head_dim"], cfg["n_qh"], cfg["n_kvh"]
        per_kv = nq // nkv
        eps, base = cfg["eps"], cfg["rope_base"]
        state = list(W["emb"][token])
        for li, L in enumerate(W["layers"]):
            a = _rms_normalise(state, L["n1"], eps)
            q = _rotate_pairs(_apply(L["wq"], a), nq, hd, pos, base)
            k = _rotate_pairs(_apply(L["wk"], a), nkv, hd, pos, base)
            v = _apply(L["wv"], a)
            self.keys[li].append(k)
            self.vals[li].append(v)
            mixed = []
            for head in range(nq):
                kvh = head // per_kv
                qh = q[head * hd:(head + 1) * hd]
                scores = []
                for kk in self.keys[li]:
                    kh = kk[kvh * hd:(kvh + 1) * hd]
                    scores.append(sum(x * y for x, y in zip(qh, kh)) / math.sqrt(hd))
                top = max(scores)
                ex = [math.exp(s - top) for s in scores]
                z = sum(ex)
                for i in range(hd):
                    acc = 0.0
                    for t, vv in enumerate(self.vals[li]):
                        acc += ex[t] / z * vv[kvh * hd + i]
                    mixed.append(acc)
            state = [s + o for s, o in zip(state, _apply(L["wo"], mixed))]
            a = _rms_normalise(state, L["n2"], eps)
            g = _apply(L["gate"], a)
            u = _apply(L["up"], a)
            hidden = [gi / (1.0 + math.exp(-gi)) * ui for gi, ui in zip(g, u)]
            state = [s + o for s, o in zip(state, _apply(L["down"], hidden))]
        return _apply(W["out"], _rms_normalise(state, W["norm"], eps))


def first_argmax(xs):
    best = 0
    for i in range(1, len(xs)):
        if xs[i] > xs[best]:
            best = i
    return best
