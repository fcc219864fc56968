"""Scalar pure-Python decode step for tiny models: an independent pin of the
oracle's vectorised NumPy step. Shares no code with oracle/ (its own format
decoders and rounding, plain loops, the math module)."""
import math
import struct


def bf16(bits):
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def e4m3(code):
    code = int(code)
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 15
    m = code & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return s * m * 2.0 ** -9
    return s * (8 + m) * 2.0 ** (e - 10)


def _rne(x, sig, min_e):
    if x == 0.0:
        return x
    m, e = math.frexp(x)
    e = max(e - 1, min_e)
    q = 2.0 ** (e - sig + 1)
    return math.copysign(round(x / q) * q, x)   # Python's round: ties to even; keep the sign of zero


def to_bf16_bits(x):
    y = _rne(x, 8, -126)
    return struct.unpack("<I", struct.pack("<f", y))[0] >> 16


def to_e4m3_code(x):
    y = max(-448.0, min(448.0, _rne(x, 4, -6)))
    neg = math.copysign(1.0, y) < 0
    a = abs(y)
    for c in range(0x7F):
        if e4m3(c) == a:
            return c | (0x80 if neg else 0)
    raise AssertionError(a)


def weight_rows(t):
    """Raw weight dict -> list of float rows."""
    w = t["w"]
    rows = []
    for n in range(w.shape[0]):
        if w.dtype.itemsize == 2:
            rows.append([bf16(v) for v in w[n]])
        else:
            s = float(t["s"][n])
            rows.append([e4m3(v) * s for v in w[n]])
    return rows


def step(weights, cfg, kv_raw, k_scale, v_scale, tokens, positions, tables, seq_lens):
    """Returns (logits rows, kv_raw) with kv_raw a nested-list copy updated in place."""
    H, d, nq, nkv, F, bs = cfg.hidden, cfg.head_dim, cfg.n_q_heads, cfg.n_kv_heads, cfg.ffn, cfg.block_size
    fp8 = kv_raw.dtype.itemsize == 1
    kvl = kv_raw.tolist()

    def kv_val(l, which, blk, h, slot, i):
        raw = kvl[l][which][blk][h][slot][i]
        sc = float((k_scale if which == 0 else v_scale)[l])
        return (e4m3(raw) if fp8 else bf16(raw)) * sc

    def norm(x, g):
        ms = sum(v * v for v in x) / len(x)
        inv = 1.0 / math.sqrt(ms + cfg.eps)
        return [x[i] * inv * g[i] for i in range(len(x))]

    def mv(rows, x):
        return [sum(r[i] * x[i] for i in range(len(x))) for r in rows]

    def rot(x, p):
        half = d // 2
        out = [0.0] * d
        for i in range(half):
            a = p * cfg.rope_theta ** (-2.0 * i / d)
            c, s = math.cos(a), math.sin(a)
            out[i] = x[i] * c - x[i + half] * s
            out[i + half] = x[i + half] * c + x[i] * s
        return out

    E = weights("embed", -1)["w"]
    W = {}
    for l in range(cfg.n_layers):
        for n in ("w_qkv", "w_o", "w_gu", "w_down"):
            W[n, l] = weight_rows(weights(n, l))
        for n in ("g_attn", "g_ffn"):
            W[n, l] = [bf16(v) for v in weights(n, l)["w"]]
    g_final = [bf16(v) for v in weights("g_final", -1)["w"]]
    lm = weight_rows(weights("lm_head", -1))

    all_logits = []
    for b in range(len(tokens)):
        r = [bf16(v) for v in E[int(tokens[b])]]
        p = int(positions[b])
        S = int(seq_lens[b])
        for l in range(cfg.n_layers):
            y = norm(r, W["g_attn", l])
            qkv = mv(W["w_qkv", l], y)
            q = [rot(qkv[h * d:(h + 1) * d], p) for h in range(nq)]
            k = [rot(qkv[(nq + h) * d:(nq + h + 1) * d], p) for h in range(nkv)]
            v = [qkv[(nq + nkv + h) * d:(nq + nkv + h + 1) * d] for h in range(nkv)]
            blk, slot = int(tables[b][p // bs]), p % bs
            for h in range(nkv):
                for i in range(d):
                    ks = k[h][i] / float(k_scale[l])
                    vs = v[h][i] / float(v_scale[l])
                    kvl[l][0][blk][h][slot][i] = to_e4m3_code(ks) if fp8 else to_bf16_bits(ks)
                    kvl[l][1][blk][h][slot][i] = to_e4m3_code(vs) if fp8 else to_bf16_bits(vs)
            o = []
            for h in range(nq):
                g = h // (nq // nkv)
                scores = []
                for t in range(S):
                    tb, ts = int(tables[b][t // bs]), t % bs
                    scores.append(sum(q[h][i] * kv_val(l, 0, tb, g, ts, i) for i in range(d)) / math.sqrt(d))
                mx = max(scores)
                ex = [math.exp(s - mx) for s in scores]
                z = sum(ex)
                acc = [0.0] * d
                for t in range(S):
                    tb, ts = int(tables[b][t // bs]), t % bs
                    for i in range(d):
                        acc[i] += ex[t] / z * kv_val(l, 1, tb, g, ts, i)
                o.extend(acc)
            dr = mv(W["w_o", l], o)
            r = [r[i] + dr[i] for i in range(H)]
            y = norm(r, W["g_ffn", l])
            gu = mv(W["w_gu", l], y)
            a = [gu[j] / (1.0 + math.exp(-gu[j])) * gu[F + j] for j in range(F)]
            dr = mv(W["w_down", l], a)
            r = [r[i] + dr[i] for i in range(H)]
        y = norm(r, g_final)
        all_logits.append(mv(lm, y))
    return all_logits, kvl
