"""ctypes binding of ``include/moe.h``: the C entry points under their own
names, taking integer device pointers and sizes.  Argument marshalling only;
every step of the layer runs in the CUDA library.  Loading fails loudly when
the library has not been built (there is no fallback path)."""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_DEVICE_CHECK = 6

MOE_F32 = 0
MOE_BF16 = 1
MOE_FWD_ONLY = 0
MOE_SAVE_FOR_BWD = 1
MOE_SHARED_READY = 2

# every symbol the header declares
EXPORTS = (
    "moe_status_string", "moe_workspace_bytes", "moe_padded_rows", "moe_route",
    "moe_permute", "moe_grouped_ffn_fwd", "moe_combine", "moe_backward",
    "moe_read_device_status", "moe_profile_enable", "moe_profile_read", "moe_permute_noalloc",
    "moe_shared_ffn_fwd", "moe_shared_backward", "moe_backward_routed", "moe_set_sm_limit",
)


class moe_dims(ctypes.Structure):
    _fields_ = [
        ("tokens", ctypes.c_int64),
        ("d_model", ctypes.c_int32),
        ("d_hidden", ctypes.c_int32),
        ("experts", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("shared_hidden", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("capacity", ctypes.c_int32),
    ]


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} (status {status})")
        self.status = status


_lib = None
_P = ctypes.c_void_p
_S = ctypes.c_size_t
_D = ctypes.POINTER(moe_dims)

_SIGS = {
    "moe_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "moe_workspace_bytes": ([_D, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
    "moe_padded_rows": ([_D, ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
    "moe_route": ([_D, _P, _P, _P, _P, _P, _P, _P, _P, _S, _P], ctypes.c_int),
    "moe_permute": ([_D, _P, _P, _P, _P, _P, _P, _S, _P], ctypes.c_int),
    "moe_grouped_ffn_fwd": ([_D, ctypes.c_int] + [_P] * 9 + [_S, _P], ctypes.c_int),
    "moe_combine": ([_D, ctypes.c_int] + [_P] * 11 + [_S, _P], ctypes.c_int),
    "moe_backward": ([_D] + [_P] * 26 + [_S, _P], ctypes.c_int),
    "moe_shared_ffn_fwd": ([_D, ctypes.c_int] + [_P] * 8 + [_S, _P], ctypes.c_int),
    "moe_shared_backward": ([_D] + [_P] * 12 + [_S, _P], ctypes.c_int),
    "moe_backward_routed": ([_D] + [_P] * 18 + [_S, _P], ctypes.c_int),
    "moe_set_sm_limit": ([ctypes.c_int], ctypes.c_int),
    "moe_read_device_status": ([_P, _S, _P, ctypes.POINTER(ctypes.c_int32)], ctypes.c_int),
    "moe_profile_enable": ([ctypes.c_int], ctypes.c_int),
    "moe_permute_noalloc": ([_D, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "moe_profile_read": ([ctypes.c_int, ctypes.c_char_p, ctypes.POINTER(ctypes.c_int64),
                          ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)],
                         ctypes.c_int),
}


def load(path: str = LIB_PATH):
    """Load the library (once).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run dropless_mixture_experts_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (args, res) in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoEError(status, where)


def make_dims(tokens, d_model, d_hidden, experts, top_k, shared_hidden=0, dtype=MOE_BF16,
              capacity=0):
    return moe_dims(int(tokens), int(d_model), int(d_hidden), int(experts), int(top_k),
                    int(shared_hidden), int(dtype), int(capacity))


def _p(v):
    return None if v in (None, 0) else ctypes.c_void_p(int(v))


def moe_workspace_bytes(dims: moe_dims, mode: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load().moe_workspace_bytes(ctypes.byref(dims), int(mode), ctypes.byref(out)),
           "moe_workspace_bytes")
    return out.value


def moe_padded_rows(dims: moe_dims) -> int:
    out = ctypes.c_int64(0)
    _check(load().moe_padded_rows(ctypes.byref(dims), ctypes.byref(out)), "moe_padded_rows")
    return out.value


def moe_route(dims, x, w_router, logits_in, logits_out, topk_idx, gates, ws, ws_bytes, stream,
              check=True, router_bias=None):
    s = load().moe_route(ctypes.byref(dims), _p(x), _p(w_router), _p(router_bias), _p(logits_in),
                         _p(logits_out), _p(topk_idx), _p(gates), _p(ws), ws_bytes, _p(stream))
    if check:
        _check(s, "moe_route")
    return s


def moe_permute(dims, topk_idx, counts, offsets, perm, inv_perm, ws, ws_bytes, stream,
                check=True):
    s = load().moe_permute(ctypes.byref(dims), _p(topk_idx), _p(counts), _p(offsets), _p(perm),
                           _p(inv_perm), _p(ws), ws_bytes, _p(stream))
    if check:
        _check(s, "moe_permute")
    return s


def moe_grouped_ffn_fwd(dims, mode, x, gates, w_gate, w_up, w_down, h_buf, a_gate_saved,
                        a_up_saved, ws, ws_bytes, stream, check=True):
    s = load().moe_grouped_ffn_fwd(ctypes.byref(dims), int(mode), _p(x), _p(gates), _p(w_gate),
                                   _p(w_up), _p(w_down), _p(h_buf), _p(a_gate_saved),
                                   _p(a_up_saved), _p(ws), ws_bytes, _p(stream))
    if check:
        _check(s, "moe_grouped_ffn_fwd")
    return s


def moe_combine(dims, mode, x, ws_gate, ws_up, ws_down, y, hs_buf, as_gate_saved, as_up_saved,
                upstream, loss, ws, ws_bytes, stream, check=True):
    s = load().moe_combine(ctypes.byref(dims), int(mode), _p(x), _p(ws_gate), _p(ws_up),
                           _p(ws_down), _p(y), _p(hs_buf), _p(as_gate_saved), _p(as_up_saved),
                           _p(upstream), _p(loss), _p(ws), ws_bytes, _p(stream))
    if check:
        _check(s, "moe_combine")
    return s


def moe_backward(dims, dy, x, w_router, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, topk_idx,
                 gates, a_gate_saved, a_up_saved, h_saved, as_gate_saved, as_up_saved, hs_saved,
                 dx, dw_router, dw_gate, dw_up, dw_down, dws_gate, dws_up, dws_down, ws, ws_bytes,
                 stream, check=True):
    args = [dy, x, w_router, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, topk_idx, gates,
            a_gate_saved, a_up_saved, h_saved, as_gate_saved, as_up_saved, hs_saved, dx,
            dw_router, dw_gate, dw_up, dw_down, dws_gate, dws_up, dws_down, ws]
    s = load().moe_backward(ctypes.byref(dims), *[_p(a) for a in args], ws_bytes, _p(stream))
    if check:
        _check(s, "moe_backward")
    return s


def moe_shared_ffn_fwd(dims, mode, x, ws_gate, ws_up, ws_down, hs_buf, as_gate_saved, as_up_saved,
                       ws, ws_bytes, stream, check=True):
    s = load().moe_shared_ffn_fwd(ctypes.byref(dims), int(mode), _p(x), _p(ws_gate), _p(ws_up),
                                  _p(ws_down), _p(hs_buf), _p(as_gate_saved), _p(as_up_saved),
                                  _p(ws), ws_bytes, _p(stream))
    if check:
        _check(s, "moe_shared_ffn_fwd")
    return s


def moe_shared_backward(dims, dy, x, ws_gate, ws_up, ws_down, as_gate_saved, as_up_saved,
                        hs_saved, dws_gate, dws_up, dws_down, ws, ws_bytes, stream, check=True):
    args = [dy, x, ws_gate, ws_up, ws_down, as_gate_saved, as_up_saved, hs_saved, dws_gate,
            dws_up, dws_down, ws]
    s = load().moe_shared_backward(ctypes.byref(dims), *[_p(a) for a in args], ws_bytes,
                                   _p(stream))
    if check:
        _check(s, "moe_shared_backward")
    return s


def moe_backward_routed(dims, dy, x, w_router, w_gate, w_up, w_down, topk_idx, gates,
                        a_gate_saved, a_up_saved, h_saved, dx, dw_router, dw_gate, dw_up,
                        dw_down, shared_done, ws, ws_bytes, stream, check=True):
    args = [dy, x, w_router, w_gate, w_up, w_down, topk_idx, gates, a_gate_saved, a_up_saved,
            h_saved, dx, dw_router, dw_gate, dw_up, dw_down, shared_done, ws]
    s = load().moe_backward_routed(ctypes.byref(dims), *[_p(a) for a in args], ws_bytes,
                                   _p(stream))
    if check:
        _check(s, "moe_backward_routed")
    return s


def moe_set_sm_limit(sms: int):
    """Caps the SMs the calling thread's later persistent launches may fill
    (0: all); see include/moe.h."""
    _check(load().moe_set_sm_limit(int(sms)), "moe_set_sm_limit")


def moe_read_device_status(ws, ws_bytes, stream):
    detail = ctypes.c_int32(0)
    s = load().moe_read_device_status(_p(ws), ws_bytes, _p(stream), ctypes.byref(detail))
    return s, detail.value


def moe_profile_enable(enable: bool):
    _check(load().moe_profile_enable(1 if enable else 0), "moe_profile_enable")


def moe_profile_read(max_entries: int = 64):
    """{kernel name: (launches, total device ms)} of the records so far."""
    names = ctypes.create_string_buffer(64 * max_entries)
    launches = (ctypes.c_int64 * max_entries)()
    ms = (ctypes.c_double * max_entries)()
    n = ctypes.c_int(0)
    _check(load().moe_profile_read(max_entries, names, launches, ms, ctypes.byref(n)),
           "moe_profile_read")
    out = {}
    for i in range(min(n.value, max_entries)):
        nm = names.raw[64 * i:64 * (i + 1)].split(b"\0", 1)[0].decode()
        out[nm] = (int(launches[i]), float(ms[i]))
    return out


def moe_permute_noalloc(dims, topk_idx, counts, offsets, perm, inv_perm, stream, check=True):
    """The counting sort of moe_permute without a workspace, for callers that
    cannot allocate device memory (its scratch is a fixed array inside the
    library; see include/moe.h for the size limit and the sharing rules)."""
    s = load().moe_permute_noalloc(ctypes.byref(dims), _p(topk_idx), _p(counts), _p(offsets),
                                   _p(perm), _p(inv_perm), _p(stream))
    if check:
        _check(s, "moe_permute_noalloc")
    return s
