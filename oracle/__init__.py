"""fp64 CPU oracle for VerKV's decode-time hot path -- TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs of
bench.py may import this package.  The CUDA library never imports, links or calls it, and it
never imports the CUDA library.  The arithmetic lives in verkv_oracle.c (plain serial fp64 C);
this module only marshals numpy arrays, widens bf16 inputs exactly to fp64 and strings the
per-head functions together in the order of "Verify Before You Fetch: Reliable KV Cache
Compression for LLM Inference" (summary page, Methodology and KVFETCH steps 1-5).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

VO_OK, VO_EINVAL, VO_EBUDGET, VO_ENOMEM = 0, 1, 2, 3

_dp = ctypes.POINTER(ctypes.c_double)
_fp = ctypes.POINTER(ctypes.c_float)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_i64p = ctypes.POINTER(ctypes.c_int64)


def lib():
    """Load (building if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.vo_philox4x32_10.argtypes = [_u32p, _u32p, _u32p]
        L.vo_philox4x32_10.restype = None
        L.vo_uniform24.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                                   ctypes.c_uint32, ctypes.c_uint64]
        L.vo_uniform24.restype = ctypes.c_double
        L.vo_poissoncomp.argtypes = [_fp, ctypes.c_int64, ctypes.c_double, ctypes.c_int64,
                                     ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32,
                                     ctypes.c_uint32, ctypes.c_uint32, _dp, _fp, _fp, _u8p,
                                     _i64p]
        L.vo_poissoncomp.restype = ctypes.c_int
        L.vo_logits.argtypes = [_dp, _dp, ctypes.c_int64, ctypes.c_int, _dp]
        L.vo_logits.restype = None
        L.vo_dense.argtypes = [_dp, _dp, ctypes.c_int64, ctypes.c_int, _dp]
        L.vo_dense.restype = None
        L.vo_certify.argtypes = [_dp, _fp, _u8p, ctypes.c_int64, ctypes.c_double,
                                 ctypes.c_double, _dp, _i64p, _dp, _dp, _u8p, _i64p, _dp]
        L.vo_certify.restype = ctypes.c_int
        L.vo_certify_cand.argtypes = [_dp, _fp, _u8p, ctypes.c_int64, ctypes.c_double,
                                      ctypes.c_double, _u8p, _dp, _i64p, _dp, _dp, _u8p, _i64p,
                                      _dp, _i64p]
        L.vo_certify_cand.restype = ctypes.c_int
        L.vo_refine.argtypes = [_dp, _dp, _fp, _u8p, _u8p, _dp, ctypes.c_double,
                                ctypes.c_int64, ctypes.c_int, _dp]
        L.vo_refine.restype = None
        L.vo_f16_round.argtypes = [ctypes.c_double, ctypes.c_int]
        L.vo_f16_round.restype = ctypes.c_double
        L.vo_f16_bits.argtypes = [ctypes.c_double]
        L.vo_f16_bits.restype = ctypes.c_uint16
        L.vo_f16_value.argtypes = [ctypes.c_uint16]
        L.vo_f16_value.restype = ctypes.c_double
        L.vo_q2_row_bytes.argtypes = [ctypes.c_int]
        L.vo_q2_row_bytes.restype = ctypes.c_int
        L.vo_q2_build.argtypes = [_fp, ctypes.c_int64, ctypes.c_int, _u8p, _dp]
        L.vo_q2_build.restype = None
        _lib = L
    return _lib


def _ptr(a, t):
    return a.ctypes.data_as(t)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class OracleError(RuntimeError):
    pass


# ------------------------------------------------------------------------------------------------
def bf16_to_f64(u16):
    """Widen bf16 bit patterns (uint16) exactly to fp64."""
    u16 = np.asarray(u16, dtype=np.uint16)
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def philox4x32_10(ctr, key):
    """One Philox4x32-10 block: ctr = 4 uint32 words, key = 2 uint32 words -> 4 uint32 words."""
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().vo_philox4x32_10(_ptr(c, _u32p), _ptr(k, _u32p), _ptr(out, _u32p))
    return out


def uniform24(seed, seq, layer, head, i):
    return lib().vo_uniform24(seed, seq, layer, head, i)


def poissoncomp(tau, eta, n_sink, n_local, seed, seq=0, layer=0, head=0):
    """PoissonComp for one head.  Returns dict(c_exact, c32, r32[n], resident[n] bool, count)."""
    tau = _c(tau, np.float32)
    n = tau.shape[0]
    r32 = np.zeros(n, dtype=np.float32)
    res = np.zeros(n, dtype=np.uint8)
    c_exact = ctypes.c_double()
    c32 = ctypes.c_float()
    count = ctypes.c_int64()
    st = lib().vo_poissoncomp(_ptr(tau, _fp), n, float(eta), int(n_sink), int(n_local),
                              int(seed), int(seq), int(layer), int(head),
                              ctypes.byref(c_exact), ctypes.byref(c32), _ptr(r32, _fp),
                              _ptr(res, _u8p), ctypes.byref(count))
    if st != VO_OK:
        raise OracleError(f"vo_poissoncomp status {st}")
    return dict(c_exact=c_exact.value, c32=np.float32(c32.value), r32=r32,
                resident=res.astype(bool), count=int(count.value))


def logits(q, keys):
    """s_i = q . k_i / sqrt(d) in fp64; q [d], keys [n][d] (fp64)."""
    q = _c(q, np.float64)
    keys = _c(keys, np.float64)
    n, d = keys.shape
    s = np.zeros(n, dtype=np.float64)
    lib().vo_logits(_ptr(q, _dp), _ptr(keys, _dp), n, d, _ptr(s, _dp))
    return s


def f16_round(x, direction):
    """The binary16 value next to x: direction < 0 the largest <= x, > 0 the smallest >= x."""
    return lib().vo_f16_round(float(x), int(direction))


def f16_bits(v):
    return int(lib().vo_f16_bits(float(v)))


def f16_value(h):
    return lib().vo_f16_value(int(h))


def q2_row_bytes(d):
    return int(lib().vo_q2_row_bytes(int(d)))


def q2_sketch(keys_bf16):
    """The 2-bit sketch of bf16 keys [n][d] (uint16 bits): (rows uint8 [n][row bytes],
    k-hat float64 [n][d], the exact dequantised keys the certificate scores)."""
    kf = np.ascontiguousarray(bf16_to_f64(keys_bf16), dtype=np.float32)
    n, d = kf.shape
    rows = np.zeros((n, q2_row_bytes(d)), dtype=np.uint8)
    khat = np.zeros((n, d), dtype=np.float64)
    lib().vo_q2_build(_ptr(kf, _fp), n, d, _ptr(rows, _u8p), _ptr(khat, _dp))
    return rows, khat


def dense(s, values):
    """Dense attention over all tokens: dict(m, D, N[d], o[d])."""
    s = _c(s, np.float64)
    values = _c(values, np.float64)
    n, d = values.shape
    out = np.zeros(2 + 2 * d, dtype=np.float64)
    lib().vo_dense(_ptr(s, _dp), _ptr(values, _dp), n, d, _ptr(out, _dp))
    return dict(m=out[0], D=out[1], N=out[2:2 + d].copy(), o=out[2 + d:].copy())


def certify(s_hat, r32, resident, eps, delta):
    """KVFetch certificate and selection for one query head (see verkv_oracle.c vo_certify)."""
    s_hat = _c(s_hat, np.float64)
    r32 = _c(r32, np.float32)
    res = _c(resident, np.uint8)
    n = s_hat.shape[0]
    nl = int(np.count_nonzero(r32 < 1.0))
    scal = np.zeros(8, dtype=np.float64)
    ints = np.zeros(4, dtype=np.int64)
    lam = np.zeros(n, dtype=np.float64)
    g = np.zeros(n, dtype=np.float64)
    F = np.zeros(n, dtype=np.uint8)
    order = np.zeros(max(nl, 1), dtype=np.int64)
    eps_k = np.zeros(nl + 1, dtype=np.float64)
    st = lib().vo_certify(_ptr(s_hat, _dp), _ptr(r32, _fp), _ptr(res, _u8p), n, float(eps),
                          float(delta), _ptr(scal, _dp), _ptr(ints, _i64p), _ptr(lam, _dp),
                          _ptr(g, _dp), _ptr(F, _u8p), _ptr(order, _i64p), _ptr(eps_k, _dp))
    if st != VO_OK:
        raise OracleError(f"vo_certify status {st}")
    return dict(m=scal[0], D=scal[1], beta=scal[2], V=scal[3], b=scal[4], l_delta=scal[5],
                eps_L=scal[6], eps_final=scal[7], certified=bool(ints[0]), k_star=int(ints[1]),
                n_L=int(ints[2]), n_fetch=int(ints[3]), lam=lam, g=g, F=F.astype(bool),
                order=order[:nl], eps_k=eps_k)


def certify_cand(s_hat, r32, resident, eps, delta, cand):
    """KVFetch certificate and selection with only the tokens of L in the mask `cand` fetchable
    (the shortlist variant; see verkv_oracle.c vo_certify_cand).  Returns certify()'s dict with
    `order` and `eps_k` over the candidates, plus `exhausted` (every candidate taken and the
    certificate still not met)."""
    s_hat = _c(s_hat, np.float64)
    r32 = _c(r32, np.float32)
    res = _c(resident, np.uint8)
    cm = _c(cand, np.uint8)
    n = s_hat.shape[0]
    nc = int(np.count_nonzero((r32 < 1.0) & (cm != 0)))
    scal = np.zeros(8, dtype=np.float64)
    ints = np.zeros(4, dtype=np.int64)
    lam = np.zeros(n, dtype=np.float64)
    g = np.zeros(n, dtype=np.float64)
    F = np.zeros(n, dtype=np.uint8)
    order = np.zeros(max(nc, 1), dtype=np.int64)
    eps_k = np.zeros(nc + 1, dtype=np.float64)
    exh = np.zeros(1, dtype=np.int64)
    st = lib().vo_certify_cand(_ptr(s_hat, _dp), _ptr(r32, _fp), _ptr(res, _u8p), n, float(eps),
                               float(delta), _ptr(cm, _u8p), _ptr(scal, _dp), _ptr(ints, _i64p),
                               _ptr(lam, _dp), _ptr(g, _dp), _ptr(F, _u8p), _ptr(order, _i64p),
                               _ptr(eps_k, _dp), _ptr(exh, _i64p))
    if st != VO_OK:
        raise OracleError(f"vo_certify_cand status {st}")
    return dict(m=scal[0], D=scal[1], beta=scal[2], V=scal[3], b=scal[4], l_delta=scal[5],
                eps_L=scal[6], eps_final=scal[7], certified=bool(ints[0]), k_star=int(ints[1]),
                n_L=int(ints[2]), n_fetch=int(ints[3]), lam=lam, g=g, F=F.astype(bool),
                order=order[:nc], eps_k=eps_k, exhausted=bool(exh[0]))


def shortlist(s_hat_heads, r32, size):
    """The per-KV-head shortlist (our reading of the pages' "128-token shortlist per KV head"):
    the `size` tokens of L (r < 1) with the largest sketch logit over the KV head's query heads,
    ties to the lower token id.  s_hat_heads [G][n] -> bool mask [n]."""
    key = np.max(np.asarray(s_hat_heads, dtype=np.float64), axis=0)
    L = np.nonzero(np.asarray(r32) < 1.0)[0]
    order = L[np.lexsort((L, -key[L]))]  # key descending, then id ascending
    mask = np.zeros(key.shape[0], dtype=bool)
    mask[order[:size]] = True
    return mask


def refine(s, values, r32, resident, F, lam, m):
    """Returned estimator after fetching: dict(D_hat, M2, lse, N_hat[d], o[d])."""
    s = _c(s, np.float64)
    values = _c(values, np.float64)
    r32 = _c(r32, np.float32)
    res = _c(resident, np.uint8)
    F = _c(F, np.uint8)
    lam = _c(lam, np.float64)
    n, d = values.shape
    out = np.zeros(3 + 2 * d, dtype=np.float64)
    lib().vo_refine(_ptr(s, _dp), _ptr(values, _dp), _ptr(r32, _fp), _ptr(res, _u8p),
                    _ptr(F, _u8p), _ptr(lam, _dp), float(m), n, d, _ptr(out, _dp))
    return dict(D_hat=out[0], M2=out[1], lse=out[2], N_hat=out[3:3 + d].copy(),
                o=out[3 + d:].copy())


# ------------------------------------------------------------------------------------------------
def attend_unit(q_heads, sketch_keys, keys, values, r32, resident, eps, delta, shortlist_size=0,
                cand=None):
    """KVFetch + refine for one KV head shared by G query heads (GQA).

    shortlist_size > 0 restricts what may be fetched to the KV head's shortlist (shortlist());
    `cand` gives that mask directly instead (e.g. the GPU's, to compare the rest given it).

    q_heads [G][d], sketch_keys [n][d] (the sketch; equal to keys for the exact sketch),
    keys/values [n][d] (the full cache), all fp64.  Each query head certifies and fetches on its
    own; the rows that move for the KV head are the union over its query heads of F \\ S, in
    ascending token id (our reading of GQA: certificates per query head, transfers per KV head).
    Returns dict(heads=[per-head dicts: cert, est, s], fetch_ids=int64[], cand, values, r32,
    resident).
    """
    heads = []
    union = np.zeros(keys.shape[0], dtype=bool)
    s_hats = [logits(q, sketch_keys) for q in q_heads]
    if cand is None and shortlist_size > 0:
        cand = shortlist(s_hats, r32, shortlist_size)
    for q, s_hat in zip(q_heads, s_hats):
        if cand is None:
            cert = certify(s_hat, r32, resident, eps, delta)
        else:
            cert = certify_cand(s_hat, r32, resident, eps, delta, cand)
        s = s_hat if sketch_keys is keys else logits(q, keys)
        est = refine(s, values, r32, resident, cert["F"], cert["lam"], cert["m"])
        union |= cert["F"] & ~np.asarray(resident, dtype=bool)
        heads.append(dict(cert=cert, est=est, s=s))
    # The exact logits s of each head and the unit's values, r and resident set stay with the
    # result so that refine() can be re-run for another fetch set F.
    return dict(heads=heads, fetch_ids=np.nonzero(union)[0].astype(np.int64), cand=cand,
                values=values, r32=r32, resident=resident)
