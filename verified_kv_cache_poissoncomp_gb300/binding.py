"""ctypes binding of libverkv (include/verkv.h): the same names, argument marshalling only.

Every function takes plain integers for device / host addresses (e.g. ``tensor.data_ptr()``) and
raises ``VerkvError`` on a status other than VERKV_OK.  The library is loaded from this package
directory; ``lib()`` raises if it has not been built (there is no fallback).
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libverkv.so")

VERKV_OK = 0
VERKV_EINVAL = 1
VERKV_EBUDGET = 2
VERKV_ECAPACITY = 3
VERKV_ENOCONVERGE = 4
VERKV_ECUDA = 5
VERKV_ECOPY = 6
VERKV_ETIMEOUT = 7
VERKV_ESTATE = 8
VERKV_ETOOLARGE = 9
VERKV_NOALLOC_MAX_LOGITS = 1 << 22

VERKV_SKETCH_EXACT = 0
VERKV_SKETCH_Q2 = 1
VERKV_FETCH_ZEROCOPY = 0
VERKV_FETCH_MEMCPY = 1
VERKV_FETCH_KEYS = 4

EXPORTED = ["verkv_sketch_bytes", "verkv_workspace_size", "verkv_create", "verkv_destroy", "verkv_set_fetch_mode",
            "verkv_poissoncomp", "verkv_sketch_build", "verkv_attend_verified",
            "verkv_fetch_refine", "verkv_selection_bitmap", "verkv_profile_enable",
            "verkv_profile_read", "verkv_launch_counts", "verkv_kernel_name", "verkv_sync",
            "verkv_last_error", "verkv_status_string", "verkv_certify_noalloc",
            "verkv_attend_dense_host", "verkv_set_shortlist", "verkv_shortlist_bitmap",
            "verkv_profile_timeline", "verkv_test_inject", "verkv_measure_sketch_stream",
            "verkv_set_sequence_offset"]
VERKV_INJECT_COPY_FAIL, VERKV_INJECT_BETA_MAXIT, VERKV_INJECT_SCORE_STALL = 1, 2, 3
VERKV_INJECT_SELECT_GATHER = 4
# kernel ids (include/verkv.h), in launch order
(VERKV_K_PC_SOLVE, VERKV_K_PC_GATHER, VERKV_K_SKETCH, VERKV_K_SCORE, VERKV_K_CERTIFY,
 VERKV_K_PARTIAL_PIVOTAL, VERKV_K_FETCH_HOST, VERKV_K_PARTIAL_STAGED, VERKV_K_MERGE,
 VERKV_K_DENSE_HOST, VERKV_K_DENSE_MERGE, VERKV_K_SHORTLIST, VERKV_K_FETCH_COPY,
 VERKV_K_FETCH_GATHER, VERKV_K_COUNT) = range(15)
# ids that are kernels (the last two time the MEMCPY fetch's copies and host gather)
KERNEL_IDS = [k for k in range(VERKV_K_COUNT) if k not in (VERKV_K_FETCH_COPY, VERKV_K_FETCH_GATHER)]


class verkv_shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("layers", ctypes.c_int32),
                ("kv_heads", ctypes.c_int32), ("q_per_kv", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("n", ctypes.c_int32), ("cap", ctypes.c_int32)]


class verkv_hset(ctypes.Structure):
    _fields_ = [("n_sink", ctypes.c_int32), ("n_local", ctypes.c_int32)]


class verkv_pivotal(ctypes.Structure):
    _fields_ = [("ids", ctypes.c_void_p), ("r", ctypes.c_void_p), ("kv", ctypes.c_void_p),
                ("count", ctypes.c_void_p), ("resident", ctypes.c_void_p),
                ("c", ctypes.c_void_p)]


class verkv_sketch(ctypes.Structure):
    _fields_ = [("format", ctypes.c_int32), ("data", ctypes.c_void_p)]


class verkv_head_stats(ctypes.Structure):
    _fields_ = [(k, ctypes.c_float) for k in
                ["m", "D", "beta", "V", "b", "eps_hat", "eps_final", "D_hat", "M2", "lse"]] + \
               [(k, ctypes.c_int32) for k in
                ["certified", "k_star", "n_L", "n_fetch", "iters", "flags"]]


STATS_FLOAT_FIELDS = ["m", "D", "beta", "V", "b", "eps_hat", "eps_final", "D_hat", "M2", "lse"]
STATS_INT_FIELDS = ["certified", "k_star", "n_L", "n_fetch", "iters", "flags"]
assert ctypes.sizeof(verkv_head_stats) == 64


class VerkvError(RuntimeError):
    def __init__(self, status, msg=""):
        self.status = status
        super().__init__(f"{_status_name(status)}: {msg}")


_lib = None


def lib():
    """Load libverkv.so; raise if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m verified_kv_cache_poissoncomp_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        L.verkv_sketch_bytes.argtypes = [ctypes.POINTER(verkv_shape), i32]
        L.verkv_sketch_bytes.restype = sz
        L.verkv_workspace_size.argtypes = [ctypes.POINTER(verkv_shape)]
        L.verkv_workspace_size.restype = sz
        L.verkv_create.argtypes = [ctypes.POINTER(vp), ctypes.c_int, vp,
                                   ctypes.POINTER(verkv_shape), vp, sz]
        L.verkv_create.restype = ctypes.c_int
        L.verkv_destroy.argtypes = [vp]
        L.verkv_destroy.restype = None
        L.verkv_set_fetch_mode.argtypes = [vp, ctypes.c_int]
        L.verkv_set_fetch_mode.restype = ctypes.c_int
        L.verkv_set_sequence_offset.argtypes = [vp, ctypes.c_int32]
        L.verkv_set_sequence_offset.restype = ctypes.c_int
        L.verkv_poissoncomp.argtypes = [vp, vp, ctypes.c_double, verkv_hset, ctypes.c_uint64, vp,
                                        vp, ctypes.POINTER(verkv_pivotal)]
        L.verkv_poissoncomp.restype = ctypes.c_int
        L.verkv_sketch_build.argtypes = [vp, vp, i32, vp]
        L.verkv_sketch_build.restype = ctypes.c_int
        L.verkv_attend_verified.argtypes = [vp, i32, vp, ctypes.POINTER(verkv_pivotal), vp,
                                            ctypes.POINTER(verkv_sketch), ctypes.c_float,
                                            ctypes.c_float, vp, vp]
        L.verkv_attend_verified.restype = ctypes.c_int
        L.verkv_fetch_refine.argtypes = [vp, vp, vp, vp, vp, vp, vp]
        L.verkv_fetch_refine.restype = ctypes.c_int
        L.verkv_shortlist_bitmap.argtypes = [vp, vp]
        L.verkv_shortlist_bitmap.restype = ctypes.c_int
        L.verkv_set_shortlist.argtypes = [vp, i32]
        L.verkv_set_shortlist.restype = ctypes.c_int
        L.verkv_attend_dense_host.argtypes = [vp, i32, vp, vp, vp, vp]
        L.verkv_attend_dense_host.restype = ctypes.c_int
        L.verkv_selection_bitmap.argtypes = [vp, vp]
        L.verkv_selection_bitmap.restype = ctypes.c_int
        L.verkv_profile_enable.argtypes = [vp, ctypes.c_int]
        L.verkv_profile_enable.restype = ctypes.c_int
        L.verkv_profile_read.argtypes = [vp, vp, vp]
        L.verkv_profile_read.restype = ctypes.c_int
        L.verkv_profile_timeline.argtypes = [vp, ctypes.c_int64, vp, vp, vp, vp]
        L.verkv_profile_timeline.restype = ctypes.c_int
        L.verkv_test_inject.argtypes = [vp, ctypes.c_int, ctypes.c_int64]
        L.verkv_test_inject.restype = ctypes.c_int
        L.verkv_measure_sketch_stream.argtypes = [vp, ctypes.c_int32, ctypes.POINTER(verkv_sketch)]
        L.verkv_measure_sketch_stream.restype = ctypes.c_int
        L.verkv_launch_counts.argtypes = [vp, vp]
        L.verkv_launch_counts.restype = ctypes.c_int
        L.verkv_kernel_name.argtypes = [ctypes.c_int]
        L.verkv_kernel_name.restype = ctypes.c_char_p
        L.verkv_sync.argtypes = [vp]
        L.verkv_sync.restype = ctypes.c_int
        L.verkv_last_error.argtypes = [vp]
        L.verkv_last_error.restype = ctypes.c_char_p
        L.verkv_status_string.argtypes = [ctypes.c_int]
        L.verkv_status_string.restype = ctypes.c_char_p
        L.verkv_certify_noalloc.argtypes = [ctypes.c_int, vp, i32, i32, i32, i32, vp, vp, vp,
                                            ctypes.c_float, ctypes.c_float, vp, vp, vp]
        L.verkv_certify_noalloc.restype = ctypes.c_int
        _lib = L
    return _lib


def _status_name(st):
    try:
        return lib().verkv_status_string(st).decode()
    except Exception:  # noqa: BLE001 -- naming only
        return f"status {st}"


def _check(st, ctx=None):
    if st != VERKV_OK:
        msg = lib().verkv_last_error(ctx).decode() if ctx else ""
        raise VerkvError(st, msg)


# ------------------------------------------------------------------------------------------------
def verkv_sketch_bytes(shape, fmt):
    return int(lib().verkv_sketch_bytes(ctypes.byref(shape), int(fmt)))


def verkv_workspace_size(shape):
    return int(lib().verkv_workspace_size(ctypes.byref(shape)))


def verkv_create(device, stream, shape, workspace, workspace_bytes):
    ctx = ctypes.c_void_p()
    _check(lib().verkv_create(ctypes.byref(ctx), int(device), stream or None,
                              ctypes.byref(shape), workspace, int(workspace_bytes)))
    return ctx


def verkv_destroy(ctx):
    lib().verkv_destroy(ctx)


def verkv_set_fetch_mode(ctx, mode):
    _check(lib().verkv_set_fetch_mode(ctx, int(mode)), ctx)


def verkv_set_sequence_offset(ctx, seq0):
    _check(lib().verkv_set_sequence_offset(ctx, int(seq0)), ctx)


def verkv_poissoncomp(ctx, tau, eta, H, seed, kv_full, r_full, pivotal):
    _check(lib().verkv_poissoncomp(ctx, tau, float(eta), H, int(seed), kv_full, r_full,
                                   ctypes.byref(pivotal)), ctx)


def verkv_sketch_build(ctx, kv_full, fmt, sketch_out):
    _check(lib().verkv_sketch_build(ctx, kv_full, int(fmt), sketch_out), ctx)


def verkv_attend_verified(ctx, layer, q, pivotal, r_full, sketch, eps, delta,
                          fetch_ids_out=None, fetch_counts_out=None):
    _check(lib().verkv_attend_verified(ctx, int(layer), q, ctypes.byref(pivotal), r_full,
                                       ctypes.byref(sketch), float(eps), float(delta),
                                       fetch_ids_out, fetch_counts_out), ctx)


def verkv_fetch_refine(ctx, ids, counts, host_kv, o_out, lse_out=None, stats_out=None):
    _check(lib().verkv_fetch_refine(ctx, ids, counts, host_kv, o_out, lse_out, stats_out), ctx)


def verkv_set_shortlist(ctx, size):
    _check(lib().verkv_set_shortlist(ctx, int(size)), ctx)


def verkv_shortlist_bitmap(ctx, out):
    _check(lib().verkv_shortlist_bitmap(ctx, out), ctx)


def verkv_attend_dense_host(ctx, layer, q, host_kv, o_out, lse_out=None):
    _check(lib().verkv_attend_dense_host(ctx, int(layer), q, host_kv, o_out, lse_out), ctx)


def verkv_selection_bitmap(ctx, out):
    _check(lib().verkv_selection_bitmap(ctx, out), ctx)


def verkv_profile_enable(ctx, on):
    _check(lib().verkv_profile_enable(ctx, int(bool(on))), ctx)


def verkv_profile_read(ctx):
    """-> (launches int64[K], total_ms float64[K]) accumulated since the last read."""
    n = (ctypes.c_int64 * VERKV_K_COUNT)()
    t = (ctypes.c_double * VERKV_K_COUNT)()
    _check(lib().verkv_profile_read(ctx, ctypes.cast(n, ctypes.c_void_p),
                                    ctypes.cast(t, ctypes.c_void_p)), ctx)
    return list(n), list(t)


def verkv_profile_timeline(ctx, max_records=1 << 16):
    """-> list of (kernel id, start ms, end ms) of the launches recorded since the last
    verkv_profile_read, times from the first record's start; the records are kept."""
    k = (ctypes.c_int32 * max_records)()
    a = (ctypes.c_double * max_records)()
    b = (ctypes.c_double * max_records)()
    n = ctypes.c_int64()
    _check(lib().verkv_profile_timeline(ctx, max_records, ctypes.cast(k, ctypes.c_void_p),
                                        ctypes.cast(a, ctypes.c_void_p),
                                        ctypes.cast(b, ctypes.c_void_p), ctypes.byref(n)), ctx)
    return [(int(k[i]), float(a[i]), float(b[i])) for i in range(n.value)]


def verkv_test_inject(ctx, what, value):
    """Failure injection for tests (VERKV_INJECT_*; see include/verkv.h)."""
    _check(lib().verkv_test_inject(ctx, int(what), int(value)), ctx)


def verkv_measure_sketch_stream(ctx, layer, sketch):
    """Stream the layer's exact sketch rows through the scoring kernel's copy ring, no arithmetic."""
    _check(lib().verkv_measure_sketch_stream(ctx, int(layer), ctypes.byref(sketch)), ctx)


def verkv_launch_counts(ctx):
    n = (ctypes.c_int64 * VERKV_K_COUNT)()
    _check(lib().verkv_launch_counts(ctx, ctypes.cast(n, ctypes.c_void_p)), ctx)
    return list(n)


def verkv_kernel_name(k):
    return lib().verkv_kernel_name(int(k)).decode()


def verkv_sync(ctx):
    _check(lib().verkv_sync(ctx), ctx)


def verkv_sync_status(ctx):
    """verkv_sync returning the raw status instead of raising."""
    return int(lib().verkv_sync(ctx))


def verkv_last_error(ctx):
    return lib().verkv_last_error(ctx).decode()


def verkv_status_string(status):
    return lib().verkv_status_string(int(status)).decode()


def verkv_certify_noalloc(device, stream, units, q_per_kv, head_dim, n, q, sketch, r_full, eps,
                          delta, stats_out, F_out, err_out):
    """The certificate and selection without a context or any allocation (logits in the
    library's fixed scratch); raises VerkvError, e.g. VERKV_ETOOLARGE above its size limit."""
    _check(lib().verkv_certify_noalloc(int(device), stream or None, int(units), int(q_per_kv),
                                       int(head_dim), int(n), q, sketch, r_full, float(eps),
                                       float(delta), stats_out, F_out, err_out))
