"""Independent numpy restatements used to pin the oracle (tests only)."""
import numpy as np


def h2f(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1(codes):
    codes = np.asarray(codes).astype(np.int64)
    return np.where(codes & 8, -1.0, 1.0) * E2M1[codes & 7]


def dequant_page(kc, vc, km, vm, is_int2, fp4=False):
    """Canonical page block -> (K^, V^) fp32 [32][128]; fmaf(code, s, z) via exact fp64
    (fp4: s * E2M1 value of the code)."""
    km = np.asarray(km).reshape(-1, 2)
    vm = np.asarray(vm).reshape(32, 4, 2)
    grp = np.arange(128) // 32
    if fp4:
        kmm = km.reshape(32, 4, 2)
        K = (e2m1(kc) * h2f(kmm[:, grp, 0])).astype(np.float32)
        V = (e2m1(vc) * h2f(vm[:, grp, 0])).astype(np.float32)
        return K, V
    if is_int2:
        ks, kz = h2f(km[:, 0])[None, :], h2f(km[:, 1])[None, :]            # per channel
    else:
        kmm = km.reshape(32, 4, 2)
        ks, kz = h2f(kmm[:, grp, 0]), h2f(kmm[:, grp, 1])                  # per token group
    vs, vz = h2f(vm[:, grp, 0]), h2f(vm[:, grp, 1])
    K = (kc.astype(np.float64) * ks + kz).astype(np.float32)
    V = (vc.astype(np.float64) * vs + vz).astype(np.float32)
    return K, V


def attention_from_export(ex, sel_index, q_row, scale, fp4_pages=None):
    """Plain fp64 softmax attention of one q row over one exported request/head
    (fp4_pages: per page, True for an FP4 page)."""
    logits, vals = [], []
    for i in range(ex["ids"].size):
        K, V = dequant_page(ex["kc"][i, sel_index], ex["vc"][i, sel_index], ex["km"][i, sel_index],
                            ex["vm"][i, sel_index], bool(ex["is_int2"][i]),
                            fp4=bool(fp4_pages[i]) if fp4_pages is not None else False)
        for s in range(int(ex["fill"][i])):
            if (int(ex["live"][i]) >> s) & 1:
                logits.append(scale * float(np.dot(q_row.astype(np.float64), K[s].astype(np.float64))))
                vals.append(V[s].astype(np.float64))
            else:
                logits.append(-1e4)
                vals.append(np.zeros(128))
    if not logits:
        return np.zeros(128)
    lg = np.array(logits)
    w = np.exp(lg - lg.max())
    return (w[:, None] * np.array(vals)).sum(0) / w.sum()


def quant_tokens_np(x, bits):
    """Uniform per-token asymmetric quantization at `bits` (2..4), fp32 numpy
    arithmetic, G = 32.  x: fp32 [T][128] -> fp32 dequantized [T][128]."""
    qmax = (1 << bits) - 1
    x = x.astype(np.float32).reshape(-1, 4, 32)
    mn = x.min(axis=2, keepdims=True)
    mx = x.max(axis=2, keepdims=True)
    s32 = ((mx - mn).astype(np.float32) / np.float32(qmax)).astype(np.float32)
    sf = s32.astype(np.float16).astype(np.float32)
    zf = mn.astype(np.float16).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        u = ((x - zf).astype(np.float32) / sf).astype(np.float32)
    c = np.where(sf == 0, 0, np.clip(np.rint(u), 0, qmax))
    xh = (c.astype(np.float64) * sf.astype(np.float64) + zf.astype(np.float64)).astype(np.float32)
    return xh.reshape(-1, 128)


def quant_int4_tokens_np(x):
    """Uniform per-token INT4 quantization (quant_tokens_np at 4 bits)."""
    return quant_tokens_np(x, 4)


def quant_fp4_tokens_np(x):
    """Uniform per-token FP4 (E2M1) quantization, G = 32, symmetric scale
    max|x| / 6 in binary16, values by nearest E2M1 level of x / s with ties
    to the even mantissa (midpoints decided by comparisons).  x: fp32 [T][128]
    -> fp32 dequantized [T][128]."""
    x = x.astype(np.float32).reshape(-1, 4, 32)
    amax = np.abs(x).max(axis=2, keepdims=True)
    sf = (amax / np.float32(6)).astype(np.float32).astype(np.float16).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        u = (x / sf).astype(np.float32)
    a = np.abs(u).astype(np.float64)
    # midpoints 0.25 .. 5; a tie goes to the level with mantissa 0 (0, 1, 2, 4)
    lv = np.select([a <= 0.25, a < 0.75, a <= 1.25, a < 1.75, a <= 2.5, a < 3.5, a <= 5.0],
                   [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0], 6.0)
    val = np.where(sf == 0, 0.0, np.where(u < 0, -lv, lv))
    return (val * sf.astype(np.float64)).astype(np.float32).reshape(-1, 128)
