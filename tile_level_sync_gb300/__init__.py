"""Python binding of the tile-level synchronisation library (include/cusync.h).

Argument marshalling only: every function forwards to the C ABI function of the same
name in the in-tree ``libcusync.so``; all computation runs in the library's CUDA
kernels.  Tensors may be passed as torch tensors (their ``data_ptr()`` is used) or as
raw integer device addresses; streams as ``torch.cuda.Stream``, a raw handle, or
``None`` for the current torch stream.  Loading fails loudly when the library is
missing: there is no fallback path.
"""

import ctypes
import os

from . import _build

c_i32, c_i64, c_u32, c_u64, c_dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_double

# ---------------------------------------------------------------- enums (cusync.h)
POLICY_STREAM, POLICY_ROW, POLICY_TILE, POLICY_STRIDED_TILE, POLICY_SENTINEL, POLICY_AUTO = range(6)
CHAIN_MLP_GELU, CHAIN_MLP_SWIGLU, CHAIN_CONV_RELU, CHAIN_ATTENTION, CHAIN_CONV_STACK = range(5)
LAUNCH_PERSISTENT, LAUNCH_PDL = range(2)
(OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_NOMEM, ERR_TIMEOUT, ERR_DEVICE) = range(7)
FLAG_NO_REORDER = 1 << 0
FLAG_TRACE = 1 << 1
FLAG_NO_RUN_OVERLAP = 1 << 2
DEBUG_SKIP_POST = 1 << 8
DEBUG_SKIP_INIT = 1 << 9
DEBUG_SKIP_SPLIT = 1 << 10
NOALLOC_MAX_SEMAPHORES = 16336

POLICY_NAMES = {"STREAM": POLICY_STREAM, "ROW": POLICY_ROW, "TILE": POLICY_TILE,
                "STRIDED": POLICY_STRIDED_TILE, "SENTINEL": POLICY_SENTINEL, "AUTO": POLICY_AUTO}


class cusync_chain_desc_t(ctypes.Structure):
    _fields_ = [
        ("kind", c_i32), ("policy", c_i32), ("launch", c_i32), ("_pad0", c_i32),
        ("M", c_i64), ("K", c_i64), ("N1", c_i64), ("N2", c_i64),
        ("n", c_i32), ("h", c_i32), ("w", c_i32), ("c", c_i32), ("k_out", c_i32),
        ("tile_n", c_i32), ("strided_group", c_i32), ("flags", c_u32), ("num_sms", c_i32), ("raster_rows", c_i32),
        ("timeout_ns", c_u64), ("l2_prefetch", c_i32), ("cta_pair", c_i32), ("ksplit", c_i32),
        ("stages", c_i32), ("ksplit_consumer", c_i32), ("bands", c_i32), ("ksplit_skew", c_i32),
    ]


class cusync_wave_report_t(ctypes.Structure):
    _fields_ = [
        ("tbs", c_i64 * 2), ("waves", c_dbl * 2), ("waves_ceil", c_i32 * 2), ("util", c_dbl * 2),
        ("stream_waves", c_i32), ("fused_waves", c_i32), ("fused_waves_frac", c_dbl),
        ("last_wave_tbs", c_i64), ("cap", c_i32), ("occupancy", c_i32), ("num_sms", c_i32),
        ("tile_m", c_i32), ("tile_n", c_i32), ("tile_k", c_i32),
    ]


class cusync_trace_rec_t(ctypes.Structure):
    _fields_ = [("tile", c_u32), ("smid", c_u32), ("cta", c_u32), ("stage", c_u32),
                ("t_claim", c_u64), ("t_ready", c_u64), ("t_mma0", c_u64), ("t_mma1", c_u64),
                ("t_epi", c_u64), ("t_post", c_u64), ("polls", c_u32), ("reloads", c_u32),
                ("land_clk", c_u32), ("check_clk", c_u32), ("t_acc", c_u64), ("t_xchg", c_u64)]


class cusync_chain_info_t(ctypes.Structure):
    _fields_ = [
        ("m_tiles", c_i32 * 2), ("n_tiles", c_i32 * 2), ("k_blocks", c_i32 * 2), ("n_out", c_i32 * 2),
        ("tile_m", c_i32), ("tile_n", c_i32), ("tile_k", c_i32),
        ("strided_group", c_i32), ("strided_distance", c_i32), ("num_flags", c_i32),
        ("grid", c_i32 * 2), ("num_sms", c_i32), ("conv_rows_per_tile", c_i32), ("cta_pair", c_i32),
        ("policy", c_i32), ("ksplit", c_i32), ("kb_per_split", c_i32),
        ("nst", c_i32), ("m_tiles2", c_i32), ("n_tiles2", c_i32), ("k_blocks2", c_i32), ("n_out2", c_i32),
        ("grid2", c_i32), ("num_flags_pw", c_i32), ("strided_group_pw", c_i32), ("strided_distance_pw", c_i32),
        ("work_buffers", c_i32), ("work_bytes", c_i64), ("ksplit_consumer", c_i32), ("kb_per_split_consumer", c_i32),
        ("raster_rows", c_i32), ("ksplit_skew", c_i32),
    ]


class cusync_latency_model_t(ctypes.Structure):
    _fields_ = [("kblock_ns", c_dbl * 2), ("wait_kblock_ns", c_dbl), ("sentinel_kblock_ns", c_dbl),
                ("start_ns", c_dbl), ("epilogue_ns", c_dbl * 2), ("post_ns", c_dbl), ("gap_ns", c_dbl),
                ("fill_ns_per_mb", c_dbl), ("tile_ns", c_dbl), ("tile_wait_ns", c_dbl)]


class cusync_policy_prediction_t(ctypes.Structure):
    _fields_ = [("us", c_dbl * 5), ("best_sync", c_i32), ("best", c_i32), ("num_sms", c_i32)]


_VP = ctypes.c_void_p
_SIGNATURES = {
    "cusync_status_string": (ctypes.c_char_p, [c_i32]),
    "cusync_wave_stats": (c_i32, [c_i64, c_i64, c_i32, c_i32, ctypes.POINTER(cusync_wave_report_t)]),
    "cusync_plan_waves": (c_i32, [ctypes.POINTER(cusync_chain_desc_t), ctypes.POINTER(cusync_wave_report_t)]),
    "cusync_create_chain": (c_i32, [ctypes.POINTER(cusync_chain_desc_t), ctypes.POINTER(_VP)]),
    "cusync_run_mlp": (c_i32, [_VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "cusync_run_conv_chain": (c_i32, [_VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "cusync_run_conv_stack": (c_i32, [_VP, _VP, _VP, _VP, _VP, _VP]),
    "cusync_run_attention": (c_i32, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "cusync_chain_check": (c_i32, [_VP, _VP, ctypes.POINTER(c_u32), ctypes.POINTER(c_u32)]),
    "cusync_chain_reset": (c_i32, [_VP, _VP]),
    "cusync_plan_info": (c_i32, [ctypes.POINTER(cusync_chain_desc_t), ctypes.POINTER(cusync_chain_info_t)]),
    "cusync_consumer_waits": (c_i32, [ctypes.POINTER(cusync_chain_desc_t), c_i32, ctypes.POINTER(c_i32),
                                      ctypes.POINTER(c_i32), ctypes.POINTER(c_u32), c_i32, ctypes.POINTER(c_i32)]),
    "cusync_consumer_unit_waits": (c_i32, [ctypes.POINTER(cusync_chain_desc_t), c_i32, c_i32, ctypes.POINTER(c_i32),
                                           ctypes.POINTER(c_i32), ctypes.POINTER(c_u32), c_i32, ctypes.POINTER(c_i32)]),
    "cusync_producer_flag": (c_i32, [ctypes.POINTER(cusync_chain_desc_t), c_i32, c_i32, ctypes.POINTER(c_i32)]),
    "cusync_pointwise_waits": (c_i32, [ctypes.POINTER(cusync_chain_desc_t), c_i32, c_i32, ctypes.POINTER(c_i32),
                                       ctypes.POINTER(c_u32), c_i32, ctypes.POINTER(c_i32)]),
    "cusync_producer_col": (c_i32, [ctypes.POINTER(cusync_chain_desc_t), c_i32, ctypes.POINTER(c_i32)]),
    "cusync_tile_at": (c_i32, [ctypes.POINTER(cusync_chain_desc_t), c_i32, c_i32, ctypes.POINTER(c_i32),
                               ctypes.POINTER(c_i32)]),
    "cusync_run_mlp_noalloc": (c_i32, [ctypes.POINTER(cusync_chain_desc_t), _VP, _VP, _VP, _VP, _VP, _VP,
                                       ctypes.POINTER(c_u32)]),
    "cusync_chain_trace": (c_i32, [_VP, _VP, ctypes.POINTER(cusync_trace_rec_t), c_i32, ctypes.POINTER(c_i32)]),
    "cusync_default_latency_model": (c_i32, [ctypes.POINTER(cusync_chain_desc_t),
                                             ctypes.POINTER(cusync_latency_model_t)]),
    "cusync_predict_policies": (c_i32, [ctypes.POINTER(cusync_chain_desc_t), ctypes.POINTER(cusync_latency_model_t),
                                        ctypes.POINTER(cusync_policy_prediction_t)]),
    "cusync_run_mlp_bands": (c_i32, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "cusync_band_wait": (c_i32, [_VP, c_i32, _VP]),
    "cusync_band_rows": (c_i32, [ctypes.POINTER(cusync_chain_desc_t), c_i32, ctypes.POINTER(c_i64),
                                 ctypes.POINTER(c_i64)]),
    "cusync_destroy_chain": (c_i32, [_VP]),
}

_lib = None


class CusyncError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def lib_path():
    return _build.LIB_PATH


def load(build_if_missing=True):
    """Load libcusync.so (building it in-tree first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing and _build.needs_build():
        _build.build()
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status, what):
    if status != OK:
        raise CusyncError(status, what)


def status_string(status):
    return load().cusync_status_string(status).decode()


def make_desc(kind=CHAIN_MLP_GELU, policy=POLICY_ROW, launch=LAUNCH_PERSISTENT, M=0, K=0, N1=0, N2=0,
              n=0, h=0, w=0, c=0, k_out=0, tile_n=0, strided_group=0, flags=0, num_sms=0, timeout_ns=0,
              raster_rows=0, l2_prefetch=0, cta_pair=0, ksplit=0, stages=0, ksplit_consumer=0, bands=0,
              ksplit_skew=0):
    if isinstance(policy, str):
        policy = POLICY_NAMES[policy]
    return cusync_chain_desc_t(kind=kind, policy=policy, launch=launch, M=M, K=K, N1=N1, N2=N2, n=n, h=h, w=w,
                               c=c, k_out=k_out, tile_n=tile_n, strided_group=strided_group, flags=flags,
                               num_sms=num_sms, timeout_ns=timeout_ns, raster_rows=raster_rows,
                               l2_prefetch=l2_prefetch, cta_pair=cta_pair, ksplit=ksplit, stages=stages,
                               ksplit_consumer=ksplit_consumer, bands=bands, ksplit_skew=ksplit_skew)


# ---------------------------------------------------------------- the C functions


def cusync_wave_stats(tbs0, tbs1, occupancy, num_sms):
    r = cusync_wave_report_t()
    _check(load().cusync_wave_stats(tbs0, tbs1, occupancy, num_sms, ctypes.byref(r)), "cusync_wave_stats")
    return r


def cusync_plan_waves(desc):
    r = cusync_wave_report_t()
    _check(load().cusync_plan_waves(ctypes.byref(desc), ctypes.byref(r)), "cusync_plan_waves")
    return r


def cusync_plan_info(desc):
    r = cusync_chain_info_t()
    _check(load().cusync_plan_info(ctypes.byref(desc), ctypes.byref(r)), "cusync_plan_info")
    return r


def cusync_default_latency_model(desc):
    r = cusync_latency_model_t()
    _check(load().cusync_default_latency_model(ctypes.byref(desc), ctypes.byref(r)), "cusync_default_latency_model")
    return r


def cusync_predict_policies(desc, model=None):
    """Predicted microseconds per policy (indexed by POLICY_*; -1 where a policy does not
    apply), plus the fastest tile-synchronised policy and the fastest overall."""
    r = cusync_policy_prediction_t()
    m = ctypes.byref(model) if model is not None else None
    _check(load().cusync_predict_policies(ctypes.byref(desc), m, ctypes.byref(r)), "cusync_predict_policies")
    return r


def cusync_pointwise_waits(desc, m_tile, head):
    fl = (c_i32 * 3)()
    pr = (c_u32 * 3)()
    n = c_i32()
    _check(load().cusync_pointwise_waits(ctypes.byref(desc), m_tile, head, fl, pr, 3, ctypes.byref(n)),
           "cusync_pointwise_waits")
    return [(fl[i], pr[i]) for i in range(n.value)]


def cusync_consumer_waits(desc, m_tile, max_entries=4096):
    kb = (c_i32 * max_entries)()
    fl = (c_i32 * max_entries)()
    pr = (c_u32 * max_entries)()
    n = c_i32()
    _check(load().cusync_consumer_waits(ctypes.byref(desc), m_tile, kb, fl, pr, max_entries, ctypes.byref(n)),
           "cusync_consumer_waits")
    if n.value > max_entries:
        raise ValueError("more waits than max_entries")
    return [(kb[i], fl[i], pr[i]) for i in range(n.value)]


def cusync_consumer_unit_waits(desc, m_tile, unit, max_entries=4096):
    kb = (c_i32 * max_entries)()
    fl = (c_i32 * max_entries)()
    pr = (c_u32 * max_entries)()
    n = c_i32()
    _check(load().cusync_consumer_unit_waits(ctypes.byref(desc), m_tile, unit, kb, fl, pr, max_entries,
                                             ctypes.byref(n)), "cusync_consumer_unit_waits")
    if n.value > max_entries:
        raise ValueError("more waits than max_entries")
    return [(kb[i], fl[i], pr[i]) for i in range(n.value)]


def cusync_producer_flag(desc, m_tile, n_tile):
    f = c_i32()
    _check(load().cusync_producer_flag(ctypes.byref(desc), m_tile, n_tile, ctypes.byref(f)), "cusync_producer_flag")
    return f.value


def cusync_producer_col(desc, y):
    c = c_i32()
    _check(load().cusync_producer_col(ctypes.byref(desc), y, ctypes.byref(c)), "cusync_producer_col")
    return c.value


def cusync_tile_at(desc, stage, u):
    m, n = c_i32(), c_i32()
    _check(load().cusync_tile_at(ctypes.byref(desc), stage, u, ctypes.byref(m), ctypes.byref(n)), "cusync_tile_at")
    return m.value, n.value


def cusync_create_chain(desc):
    h = _VP()
    _check(load().cusync_create_chain(ctypes.byref(desc), ctypes.byref(h)), "cusync_create_chain")
    return h


def cusync_run_mlp(chain, X, W1t, W2t, H, Y, stream=None):
    _check(load().cusync_run_mlp(chain, _ptr(X), _ptr(W1t), _ptr(W2t), _ptr(H), _ptr(Y), _stream(stream)),
           "cusync_run_mlp")


def cusync_run_conv_chain(chain, x, w1, w2, y1, y2, stream=None):
    _check(load().cusync_run_conv_chain(chain, _ptr(x), _ptr(w1), _ptr(w2), _ptr(y1), _ptr(y2), _stream(stream)),
           "cusync_run_conv_chain")


def cusync_run_conv_stack(chain, x, w, work, y, stream=None):
    _check(load().cusync_run_conv_stack(chain, _ptr(x), _ptr(w), _ptr(work), _ptr(y), _stream(stream)),
           "cusync_run_conv_stack")


def cusync_run_attention(chain, X, Wqkv_t, W2t, XQKV, XDot, Y, stream=None):
    _check(load().cusync_run_attention(chain, _ptr(X), _ptr(Wqkv_t), _ptr(W2t), _ptr(XQKV), _ptr(XDot), _ptr(Y),
                                       _stream(stream)), "cusync_run_attention")


def cusync_run_mlp_noalloc(desc, X, W1t, W2t, H, Y, stream=None, wait=False):
    """Allocation-free MLP chain run (see include/cusync.h).  With wait=True it returns
    (status, device error word) after the chain finished; else it returns after launching."""
    err = c_u32() if wait else None
    st = load().cusync_run_mlp_noalloc(ctypes.byref(desc), _ptr(X), _ptr(W1t), _ptr(W2t), _ptr(H), _ptr(Y),
                                       _stream(stream), ctypes.byref(err) if wait else None)
    if st not in (OK, ERR_TIMEOUT, ERR_DEVICE):
        raise CusyncError(st, "cusync_run_mlp_noalloc")
    return st, (err.value if wait else None)


def cusync_run_mlp_bands(chain, X, W1t, W2t, H, Y, band_stream, stream=None):
    _check(load().cusync_run_mlp_bands(chain, _ptr(X), _ptr(W1t), _ptr(W2t), _ptr(H), _ptr(Y), _stream(stream),
                                       _stream(band_stream)), "cusync_run_mlp_bands")


def cusync_band_wait(chain, band, band_stream):
    _check(load().cusync_band_wait(chain, band, _stream(band_stream)), "cusync_band_wait")


def cusync_band_rows(desc, band):
    r0, n = c_i64(), c_i64()
    _check(load().cusync_band_rows(ctypes.byref(desc), band, ctypes.byref(r0), ctypes.byref(n)), "cusync_band_rows")
    return r0.value, n.value


def cusync_chain_check(chain, stream=None):
    """Return (status, code, detail); status is OK, ERR_TIMEOUT or ERR_DEVICE."""
    code, detail = c_u32(), c_u32()
    st = load().cusync_chain_check(chain, _stream(stream), ctypes.byref(code), ctypes.byref(detail))
    if st not in (OK, ERR_TIMEOUT, ERR_DEVICE):
        raise CusyncError(st, "cusync_chain_check")
    return st, code.value, detail.value


def cusync_chain_reset(chain, stream=None):
    _check(load().cusync_chain_reset(chain, _stream(stream)), "cusync_chain_reset")


def cusync_chain_trace(chain, stream=None, max_records=1 << 20):
    """Per-tile timeline of the last traced run, as a list of dicts."""
    n = c_i32()
    _check(load().cusync_chain_trace(chain, _stream(stream), None, 0, ctypes.byref(n)), "cusync_chain_trace")
    k = min(n.value, max_records)
    buf = (cusync_trace_rec_t * k)()
    _check(load().cusync_chain_trace(chain, _stream(stream), buf, k, ctypes.byref(n)), "cusync_chain_trace")
    return [{f: getattr(r, f) for f, _ in cusync_trace_rec_t._fields_} for r in buf]


def cusync_destroy_chain(chain):
    _check(load().cusync_destroy_chain(chain), "cusync_destroy_chain")


class Chain:
    """Owns a chain handle; ``run`` forwards to cusync_run_mlp / cusync_run_conv_chain."""

    def __init__(self, desc):
        self.desc = desc
        self.handle = cusync_create_chain(desc)

    def run(self, a, w1, w2, h, y, stream=None, h2=None):
        """Run the chain; h2 is the second intermediate (XDot) of an attention chain.  A
        convolution stack takes its stacked weights as w1 and its workspace as h (w2
        unused)."""
        if self.desc.kind == CHAIN_CONV_STACK:
            cusync_run_conv_stack(self.handle, a, w1, h, y, stream)
        elif self.desc.kind == CHAIN_CONV_RELU:
            cusync_run_conv_chain(self.handle, a, w1, w2, h, y, stream)
        elif self.desc.kind == CHAIN_ATTENTION:
            cusync_run_attention(self.handle, a, w1, w2, h, h2, y, stream)
        else:
            cusync_run_mlp(self.handle, a, w1, w2, h, y, stream)

    def check(self, stream=None):
        return cusync_chain_check(self.handle, stream)

    def reset(self, stream=None):
        cusync_chain_reset(self.handle, stream)

    def info(self):
        return cusync_plan_info(self.desc)

    def trace(self, stream=None):
        return cusync_chain_trace(self.handle, stream)

    def close(self):
        if self.handle is not None:
            cusync_destroy_chain(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
