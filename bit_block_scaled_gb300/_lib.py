"""ctypes binding of libmoe4 (include/moe4.h): same names, argument
marshalling only. Tensors are torch CUDA tensors (PyTorch provides device
memory and streams); every step of the layer runs in the library's kernels.
There is no fallback: if the library cannot be loaded, importing the binding
raises.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe4.so")

MOE_OK = 0
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_CUDA",
          4: "MOE_ERR_TIMEOUT", 5: "MOE_ERR_BAD_INDEX", 6: "MOE_ERR_WORKSPACE",
          7: "MOE_ERR_SCALE_RANGE"}
FMT = {"nvfp4": 0, "mxfp4": 1, "int4": 2}
ACT = {"swigluoai": 0, "relu2": 1}
ROUTE = {"topk_softmax": 0, "sigmoid_bias": 1}
LAYOUT = {"interleaved": 0, "concat": 1}
STATUS_BYTES = 256

#: symbols include/moe4.h declares
EXPORTS = ("moe_padded_rows", "moe_workspace_size", "moe_route_topk", "moe_align_permute",
           "moe_grouped_gemm1_act", "moe_grouped_gemm2_weighted", "moe_unpermute_reduce",
           "moe_forward", "moe_forward_host", "moe_read_status", "moe_clear_status", "moe_wait_selftest",
           "moe_status_string", "moe_last_launch_count", "moe_forward_static", "moe_forward_profile",
           "moe_import_gptq_int4", "moe_import_modelopt_global_scale")


class MoeError(RuntimeError):
    def __init__(self, code, where):
        super().__init__(f"{where}: {STATUS.get(code, code)}")
        self.code = code


class QWeight(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("E", ctypes.c_int32), ("N", ctypes.c_int32),
                ("K", ctypes.c_int32), ("q", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("zeros", ctypes.c_void_p), ("gscale", ctypes.c_void_p), ("bias", ctypes.c_void_p)]


class Act(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("alpha", ctypes.c_float), ("limit", ctypes.c_float)]


_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
_SIGS = {
    "moe_padded_rows": (_i64, [_i32, _i32, _i32, _i32]),
    "moe_workspace_size": (_i32, [_i32] * 6 + [ctypes.POINTER(_sz)]),
    "moe_route_topk": (_i32, [_vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp]),
    "moe_align_permute": (_i32, [_vp, _i32, _i32, _i32, _i32, _vp, _i32, _vp, _vp, _vp, _vp, _vp,
                                 _vp, _vp]),
    "moe_grouped_gemm1_act": (_i32, [_vp, _vp, _vp, _i32, _i32, ctypes.POINTER(QWeight), _i32, Act,
                                     _vp, _vp, _vp]),
    "moe_grouped_gemm2_weighted": (_i32, [_vp, _vp, _vp, _i32, ctypes.POINTER(QWeight), _vp, _i32,
                                          _i32, _vp, _vp, _vp]),
    "moe_unpermute_reduce": (_i32, [_vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp]),
    "moe_forward": (_i32, [_vp, _vp, _vp] + [_i32] * 6 + [ctypes.POINTER(QWeight)] * 2 +
                    [_i32, Act, _i32, _i32, _vp, _vp, _sz, _vp]),
    "moe_forward_host": (_i32, [_vp, _vp, _vp] + [_i32] * 6 + [ctypes.POINTER(QWeight)] * 2 +
                         [_i32, Act, _i32, _i32, _vp, _vp, _sz, _vp]),
    "moe_forward_profile": (_i32, [_vp, _vp, _vp] + [_i32] * 6 + [ctypes.POINTER(QWeight)] * 2 +
                            [_i32, Act, _i32, _i32, _vp, _vp, _sz, _vp, _vp]),
    "moe_forward_static": (_i32, [_vp, _vp, _vp] + [_i32] * 6 + [ctypes.POINTER(QWeight)] * 2 +
                           [_i32, Act, _i32, _i32, _vp, _vp, _vp]),
    "moe_read_status": (_i32, [_vp, _vp, ctypes.POINTER(_i32)]),
    "moe_clear_status": (_i32, [_vp, _vp]),
    "moe_wait_selftest": (_i32, [_vp, _vp]),
    "moe_status_string": (ctypes.c_char_p, [_i32]),
    "moe_last_launch_count": (_i32, []),
    "moe_import_gptq_int4": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp]),
    "moe_import_modelopt_global_scale": (_i32, [ctypes.c_float, _i32, _vp]),
}

_lib = None


def load(path: str = LIB_PATH):
    """Loads the library (once). Raises ImportError when it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libmoe4 is not built ({path} missing); run "
                          "bit_block_scaled_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(code, where):
    if code != MOE_OK:
        raise MoeError(code, where)


def qweight(w: dict) -> QWeight:
    """QWeight view of a projection dict of device tensors (as made by synth);
    the caller keeps the dict alive while the struct is in use."""
    return QWeight(int(w["fmt"]), int(w["q"].shape[0]), int(w["q"].shape[1]),
                   int(w["q"].shape[2] * 2), w["q"].data_ptr(), w["scales"].data_ptr(),
                   _ptr(w.get("zeros")), _ptr(w.get("gscale")), _ptr(w.get("bias")))


def act(kind="swigluoai", alpha=1.702, limit=7.0) -> Act:
    return Act(ACT[kind] if isinstance(kind, str) else int(kind), float(alpha), float(limit))


# --------------------------------------------------------------------- entry points
def moe_padded_rows(T, k, E, block_m):
    return int(load().moe_padded_rows(T, k, E, block_m))


def moe_workspace_size(T, E, k, H, I, block_m=16):
    n = ctypes.c_size_t(0)
    _check(load().moe_workspace_size(T, E, k, H, I, block_m, ctypes.byref(n)), "moe_workspace_size")
    return int(n.value)


def moe_route_topk(logits, sel_bias, k, route, topk_ids, topk_weights, ws, stream=None):
    T, E = logits.shape
    _check(load().moe_route_topk(_ptr(logits), _ptr(sel_bias), T, E, k, route, _ptr(topk_ids),
                                 _ptr(topk_weights), _ptr(ws), _stream(stream)), "moe_route_topk")


def moe_align_permute(topk_ids, E, block_m, x, sorted_token_ids, expert_offsets, block_expert_ids,
                      row_pos, x_perm, ws, stream=None):
    T, k = topk_ids.shape
    H = x.shape[1]
    _check(load().moe_align_permute(_ptr(topk_ids), T, k, E, block_m, _ptr(x), H,
                                    _ptr(sorted_token_ids), _ptr(expert_offsets),
                                    _ptr(block_expert_ids), _ptr(row_pos), _ptr(x_perm), _ptr(ws),
                                    _stream(stream)), "moe_align_permute")


def moe_grouped_gemm1_act(x_perm, sorted_token_ids, expert_offsets, num_rows, w13, gate_up_layout,
                          activation, a_out, ws, stream=None):
    qw = w13 if isinstance(w13, QWeight) else qweight(w13)
    _check(load().moe_grouped_gemm1_act(_ptr(x_perm), _ptr(sorted_token_ids), _ptr(expert_offsets),
                                        x_perm.shape[0], num_rows, ctypes.byref(qw), gate_up_layout,
                                        activation, _ptr(a_out), _ptr(ws), _stream(stream)),
           "moe_grouped_gemm1_act")


def moe_grouped_gemm2_weighted(a, sorted_token_ids, expert_offsets, w2, topk_weights_flat,
                               mul_topk_weights, num_rows, y, ws, stream=None):
    qw = w2 if isinstance(w2, QWeight) else qweight(w2)
    _check(load().moe_grouped_gemm2_weighted(_ptr(a), _ptr(sorted_token_ids), _ptr(expert_offsets),
                                             a.shape[0], ctypes.byref(qw), _ptr(topk_weights_flat),
                                             int(mul_topk_weights), num_rows, _ptr(y), _ptr(ws),
                                             _stream(stream)), "moe_grouped_gemm2_weighted")


def moe_unpermute_reduce(y, row_pos, T, k, out, ws, stream=None):
    _check(load().moe_unpermute_reduce(_ptr(y), _ptr(row_pos), T, k, y.shape[1], y.shape[0],
                                       _ptr(out), _ptr(ws), _stream(stream)), "moe_unpermute_reduce")


def moe_forward(x, logits, sel_bias, k, route, w13, w2, gate_up_layout, activation, mul_topk_weights,
                block_m, out, ws, stream=None):
    T, H = x.shape
    E = logits.shape[1]
    q13 = w13 if isinstance(w13, QWeight) else qweight(w13)
    q2 = w2 if isinstance(w2, QWeight) else qweight(w2)
    I = q2.K
    _check(load().moe_forward(_ptr(x), _ptr(logits), _ptr(sel_bias), T, E, k, H, I, route,
                              ctypes.byref(q13), ctypes.byref(q2), gate_up_layout, activation,
                              int(mul_topk_weights), block_m, _ptr(out), _ptr(ws), ws.numel(),
                              _stream(stream)), "moe_forward")


def moe_forward_host(x_host, logits_host, sel_bias, k, route, w13, w2, gate_up_layout, activation,
                     mul_topk_weights, block_m, out_host, ws, stream=None):
    T, H = x_host.shape
    E = logits_host.shape[1]
    q13 = w13 if isinstance(w13, QWeight) else qweight(w13)
    q2 = w2 if isinstance(w2, QWeight) else qweight(w2)
    _check(load().moe_forward_host(_ptr(x_host), _ptr(logits_host), _ptr(sel_bias), T, E, k, H, q2.K,
                                   route, ctypes.byref(q13), ctypes.byref(q2), gate_up_layout,
                                   activation, int(mul_topk_weights), block_m, _ptr(out_host),
                                   _ptr(ws), ws.numel(), _stream(stream)), "moe_forward_host")


def moe_forward_profile(x, logits, sel_bias, k, route, w13, w2, gate_up_layout, activation,
                        mul_topk_weights, block_m, out, ws, stream=None):
    """moe_forward plus the device time (ms) of its six kernels:
    dict(route, align, gather, gemm1, gemm2, unpermute)."""
    T, H = x.shape
    E = logits.shape[1]
    q13 = w13 if isinstance(w13, QWeight) else qweight(w13)
    q2 = w2 if isinstance(w2, QWeight) else qweight(w2)
    ms = (ctypes.c_float * 6)()
    _check(load().moe_forward_profile(_ptr(x), _ptr(logits), _ptr(sel_bias), T, E, k, H, q2.K, route,
                                      ctypes.byref(q13), ctypes.byref(q2), gate_up_layout, activation,
                                      int(mul_topk_weights), block_m, _ptr(out), _ptr(ws), ws.numel(),
                                      _stream(stream), ms), "moe_forward_profile")
    return dict(zip(("route", "align", "gather", "gemm1", "gemm2", "unpermute"), list(ms)))


def moe_forward_static(x, logits, sel_bias, k, route, w13, w2, gate_up_layout, activation,
                       mul_topk_weights, block_m, out, status_out=None, stream=None):
    """moe_forward with the library's own static device workspace (no
    workspace argument, nothing allocated); status_out: optional device
    uint32/int32 tensor that receives the raw device status word."""
    T, H = x.shape
    E = logits.shape[1]
    q13 = w13 if isinstance(w13, QWeight) else qweight(w13)
    q2 = w2 if isinstance(w2, QWeight) else qweight(w2)
    _check(load().moe_forward_static(_ptr(x), _ptr(logits), _ptr(sel_bias), T, E, k, H, q2.K, route,
                                     ctypes.byref(q13), ctypes.byref(q2), gate_up_layout, activation,
                                     int(mul_topk_weights), block_m, _ptr(out), _ptr(status_out),
                                     _stream(stream)), "moe_forward_static")


def moe_read_status(ws, stream=None):
    st = ctypes.c_int(0)
    _check(load().moe_read_status(_ptr(ws), _stream(stream), ctypes.byref(st)), "moe_read_status")
    return int(st.value)


def moe_clear_status(ws, stream=None):
    _check(load().moe_clear_status(_ptr(ws), _stream(stream)), "moe_clear_status")


def moe_wait_selftest(ws, stream=None):
    _check(load().moe_wait_selftest(_ptr(ws), _stream(stream)), "moe_wait_selftest")


def moe_status_string(code):
    return load().moe_status_string(code).decode()


def moe_last_launch_count():
    return int(load().moe_last_launch_count())


def _host_ptr(a):
    """Pointer to a C-contiguous numpy array in host memory (None stays NULL)."""
    if a is None:
        return None
    import numpy as np
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "host arrays must be C-contiguous numpy"
    return ctypes.c_void_p(a.ctypes.data)


def moe_import_gptq_int4(qweight_, qzeros, scales, g_idx=None, group_size=64, zero_offset=0):
    """GPTQ INT4 tensors of one linear layer (numpy, host) -> (q uint8 [N, K/2],
    scales fp16 [N, K/64], zeros uint8 [N, ceil(K/128)]) in the library's layout."""
    import numpy as np
    qweight_ = np.ascontiguousarray(qweight_, dtype=np.int32)
    qzeros = np.ascontiguousarray(qzeros, dtype=np.int32)
    scales = np.ascontiguousarray(scales, dtype=np.float16)
    if g_idx is not None:
        g_idx = np.ascontiguousarray(g_idx, dtype=np.int32)
    K8, N = qweight_.shape
    K = 8 * K8
    q = np.empty((N, K // 2), dtype=np.uint8)
    s_out = np.empty((N, max(K // 64, 1)), dtype=np.float16)
    z_out = np.empty((N, max((K // 64 + 1) // 2, 1)), dtype=np.uint8)
    _check(load().moe_import_gptq_int4(_host_ptr(qweight_), _host_ptr(qzeros), _host_ptr(scales),
                                       _host_ptr(g_idx), K, N, group_size, zero_offset, _host_ptr(q),
                                       _host_ptr(s_out), _host_ptr(z_out)), "moe_import_gptq_int4")
    return q, s_out, z_out


def moe_import_modelopt_global_scale(weight_scale_2, E):
    """The per-expert global scales (numpy float32 [E]) for a ModelOpt
    checkpoint's single weight_scale_2."""
    import numpy as np
    g = np.empty(E, dtype=np.float32)
    _check(load().moe_import_modelopt_global_scale(float(weight_scale_2), E, _host_ptr(g)),
           "moe_import_modelopt_global_scale")
    return g
