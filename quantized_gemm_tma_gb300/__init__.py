"""Python binding of the GB300 quantized GEMM library (``include/hq.h``).

Argument marshalling only: every function here forwards to the C ABI of the
in-tree ``libhq.so`` (built by ``_build.build()``), whose kernels do all the
work.  Pointers may be given as integers or as objects with ``data_ptr()``
(torch tensors); streams as integers, ``None`` (default stream) or objects
with a ``cuda_stream`` attribute.  A non-OK status raises ``HQError``.

There is no fallback: if the library is missing, importing the functions
raises.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libhq.so")

# enums of hq.h
HQ_OK, HQ_ERR_INVALID_ARG, HQ_ERR_UNSUPPORTED, HQ_ERR_ALIGNMENT = 0, 1, 2, 3
HQ_ERR_WORKSPACE_TOO_SMALL, HQ_ERR_CUDA, HQ_ERR_DEVICE_TIMEOUT, HQ_ERR_ARCH, HQ_ERR_INVALID_VALUE = 4, 5, 6, 7, 8
HQ_W_INT4, HQ_W_INT6, HQ_W_MXFP4, HQ_W_FP8_E4M3, HQ_W_NVFP4, HQ_W_MXINT4 = 0, 1, 2, 3, 4, 5
HQ_A_BF16, HQ_A_FP16, HQ_A_FP8_E4M3, HQ_A_MXFP8_E4M3 = 0, 1, 2, 3
HQ_S_BF16, HQ_S_FP16, HQ_S_FP32, HQ_S_UE8M0, HQ_S_E4M3 = 0, 1, 2, 3, 4
HQ_FLAG_BATCH_INVARIANT = 0x1
HQ_FLAG_NOALLOC_RESET = 0x100
HQ_MOE_GROUPED_CONTIGUOUS, HQ_MOE_GROUPED_MASKED = 0, 1

WTYPES = {"int4": HQ_W_INT4, "int6": HQ_W_INT6, "mxfp4": HQ_W_MXFP4, "fp8": HQ_W_FP8_E4M3, "nvfp4": HQ_W_NVFP4,
          "mxint4": HQ_W_MXINT4}
ATYPES = {"bf16": HQ_A_BF16, "fp16": HQ_A_FP16, "fp8": HQ_A_FP8_E4M3, "mxfp8": HQ_A_MXFP8_E4M3}
STYPES = {"bf16": HQ_S_BF16, "fp16": HQ_S_FP16, "fp32": HQ_S_FP32, "ue8m0": HQ_S_UE8M0, "e4m3": HQ_S_E4M3}

#: every symbol include/hq.h declares
EXPORTS = [
    "hq_version", "hq_status_string", "hq_transform_size", "hq_transform", "hq_untransform",
    "hq_gemm_workspace_size", "hq_workspace_init", "hq_gemm", "hq_gemm_noalloc", "hq_moe_workspace_size",
    "hq_moe_gemm", "hq_moe_ffn_workspace_size", "hq_moe_ffn", "hq_moe_grouped_workspace_size",
    "hq_moe_grouped_gemm", "hq_status_read", "hq_last_plan", "hq_plan_query", "hq_selftest_wait_timeout",
    "hq_moe_plan_query", "hq_tuning_reload", "hq_mxfp8_quantize",
]

#: size of the fixed device scratch behind hq_gemm_noalloc
HQ_NOALLOC_SCRATCH_BYTES = 8 << 20


class HQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class WeightDesc(ctypes.Structure):
    """hq_weight_desc."""
    _fields_ = [
        ("wtype", ctypes.c_int32), ("stype", ctypes.c_int32), ("n", ctypes.c_int32), ("k", ctypes.c_int32),
        ("num_experts", ctypes.c_int32), ("group_k", ctypes.c_int32), ("group_n", ctypes.c_int32),
        ("signed_codes", ctypes.c_int32), ("has_zeros", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("zeros", ctypes.c_void_p),
        ("tensor_scales", ctypes.c_void_p),
    ]


class PlanInfo(ctypes.Structure):
    """hq_plan_info."""
    _fields_ = [("bn", ctypes.c_int32), ("splits", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("launches", ctypes.c_int32), ("stages", ctypes.c_int32), ("tile_class", ctypes.c_int32),
                ("groups", ctypes.c_int32), ("x_stages", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libhq.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run quantized_gemm_tma_gb300._build.build() first")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, u32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_size_t
        dp = ctypes.POINTER(WeightDesc)
        sig = {
            "hq_version": ([], i32),
            "hq_status_string": ([i32], ctypes.c_char_p),
            "hq_transform_size": ([dp, ctypes.POINTER(sz)], i32),
            "hq_transform": ([dp, vp, sz, vp], i32),
            "hq_untransform": ([dp, vp, vp, vp, vp, vp], i32),
            "hq_gemm_workspace_size": ([dp, i32, i32, ctypes.POINTER(sz)], i32),
            "hq_workspace_init": ([vp, sz, vp], i32),
            "hq_gemm": ([dp, vp, i32, i32, vp, i64, vp, vp, i64, vp, sz, u32, vp], i32),
            "hq_gemm_noalloc": ([dp, vp, i32, i32, vp, i64, vp, vp, i64, u32, vp, vp], i32),
            "hq_moe_workspace_size": ([dp, i32, i32, i32, ctypes.POINTER(sz)], i32),
            "hq_moe_gemm": ([dp, vp, i32, i32, vp, vp, i32, vp, i64, vp, i64, vp, vp, vp, sz, u32, vp], i32),
            "hq_moe_ffn_workspace_size": ([dp, dp, i32, i32, ctypes.POINTER(sz)], i32),
            "hq_moe_ffn": ([dp, vp, dp, vp, i32, i32, vp, vp, i32, vp, i64, vp, i64, vp, sz, u32, vp], i32),
            "hq_moe_grouped_workspace_size": ([dp, i32, i32, ctypes.POINTER(sz)], i32),
            "hq_moe_grouped_gemm": ([dp, vp, i32, i32, vp, i32, i32, vp, i64, vp, i64, vp, sz, u32, vp], i32),
            "hq_status_read": ([vp, i32, vp, ctypes.POINTER(i32)], i32),
            "hq_last_plan": ([ctypes.POINTER(PlanInfo)], i32),
            "hq_plan_query": ([dp, i32, i32, i32, i64, u32, ctypes.POINTER(PlanInfo)], i32),
            "hq_selftest_wait_timeout": ([vp, vp], i32),
            "hq_moe_plan_query": ([dp, i32, i32, i32, i64, ctypes.POINTER(PlanInfo)], i32),
            "hq_tuning_reload": ([], None),
            "hq_mxfp8_quantize": ([i32, i32, vp, i64, vp, i64, vp, i64, vp], i32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _check(st: int, where: str) -> None:
    if st != HQ_OK:
        raise HQError(st, where)


def status_string(status: int) -> str:
    return lib().hq_status_string(status).decode()


def hq_version() -> int:
    return int(lib().hq_version())


def make_desc(wtype, stype, n, k, num_experts=1, group_k=128, group_n=1, signed_codes=True, has_zeros=False,
              codes=None, scales=None, zeros=None, tensor_scales=None) -> WeightDesc:
    """Build an hq_weight_desc (enum names or values accepted)."""
    return WeightDesc(WTYPES.get(wtype, wtype), STYPES.get(stype, stype), n, k, num_experts, group_k, group_n,
                      1 if signed_codes else 0, 1 if has_zeros else 0, 0,
                      _ptr(codes), _ptr(scales), _ptr(zeros), _ptr(tensor_scales))


def hq_transform_size(desc: WeightDesc) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().hq_transform_size(ctypes.byref(desc), ctypes.byref(out)), "hq_transform_size")
    return out.value


def hq_transform(desc: WeightDesc, dst, dst_bytes: int, stream=None) -> None:
    _check(lib().hq_transform(ctypes.byref(desc), _ptr(dst), dst_bytes, _stream(stream)), "hq_transform")


def hq_untransform(desc: WeightDesc, src, codes, scales, zeros=None, stream=None) -> None:
    _check(lib().hq_untransform(ctypes.byref(desc), _ptr(src), _ptr(codes), _ptr(scales), _ptr(zeros),
                                _stream(stream)), "hq_untransform")


def hq_gemm_workspace_size(desc: WeightDesc, m: int, atype) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().hq_gemm_workspace_size(ctypes.byref(desc), m, ATYPES.get(atype, atype), ctypes.byref(out)),
           "hq_gemm_workspace_size")
    return out.value


def hq_workspace_init(workspace, nbytes: int, stream=None) -> None:
    _check(lib().hq_workspace_init(_ptr(workspace), nbytes, _stream(stream)), "hq_workspace_init")


def hq_gemm(desc: WeightDesc, w_t, m: int, atype, x, ldx: int, x_scales, y, ldy: int, workspace, ws_bytes: int,
            flags: int = 0, stream=None) -> None:
    _check(lib().hq_gemm(ctypes.byref(desc), _ptr(w_t), m, ATYPES.get(atype, atype), _ptr(x), ldx, _ptr(x_scales),
                         _ptr(y), ldy, _ptr(workspace), ws_bytes, flags, _stream(stream)), "hq_gemm")


def hq_gemm_noalloc(desc: WeightDesc, w_t, m: int, atype, x, ldx: int, x_scales, y, ldy: int, flags: int = 0,
                    device_status=None, stream=None) -> None:
    _check(lib().hq_gemm_noalloc(ctypes.byref(desc), _ptr(w_t), m, ATYPES.get(atype, atype), _ptr(x), ldx,
                                 _ptr(x_scales), _ptr(y), ldy, flags, _ptr(device_status), _stream(stream)),
           "hq_gemm_noalloc")


def hq_moe_workspace_size(desc: WeightDesc, tokens: int, topk: int, atype) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().hq_moe_workspace_size(ctypes.byref(desc), tokens, topk, ATYPES.get(atype, atype),
                                       ctypes.byref(out)), "hq_moe_workspace_size")
    return out.value


def hq_moe_gemm(desc: WeightDesc, w_t, tokens: int, topk: int, topk_ids, topk_w, atype, x, ldx: int, y, ldy: int,
                expert_offsets_out, perm_out, workspace, ws_bytes: int, flags: int = 0, stream=None) -> None:
    _check(lib().hq_moe_gemm(ctypes.byref(desc), _ptr(w_t), tokens, topk, _ptr(topk_ids), _ptr(topk_w),
                             ATYPES.get(atype, atype), _ptr(x), ldx, _ptr(y), ldy, _ptr(expert_offsets_out),
                             _ptr(perm_out), _ptr(workspace), ws_bytes, flags, _stream(stream)), "hq_moe_gemm")


def hq_moe_ffn_workspace_size(w13: WeightDesc, w2: WeightDesc, tokens: int, topk: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().hq_moe_ffn_workspace_size(ctypes.byref(w13), ctypes.byref(w2), tokens, topk, ctypes.byref(out)),
           "hq_moe_ffn_workspace_size")
    return out.value


def hq_moe_ffn(w13: WeightDesc, w13_t, w2: WeightDesc, w2_t, tokens: int, topk: int, topk_ids, topk_w, atype, x,
               ldx: int, y, ldy: int, workspace, ws_bytes: int, flags: int = 0, stream=None) -> None:
    _check(lib().hq_moe_ffn(ctypes.byref(w13), _ptr(w13_t), ctypes.byref(w2), _ptr(w2_t), tokens, topk,
                            _ptr(topk_ids), _ptr(topk_w), ATYPES.get(atype, atype), _ptr(x), ldx, _ptr(y), ldy,
                            _ptr(workspace), ws_bytes, flags, _stream(stream)), "hq_moe_ffn")


def hq_moe_grouped_workspace_size(desc: WeightDesc, form: int, rows: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().hq_moe_grouped_workspace_size(ctypes.byref(desc), form, rows, ctypes.byref(out)),
           "hq_moe_grouped_workspace_size")
    return out.value


def hq_moe_grouped_gemm(desc: WeightDesc, w_t, form: int, rows: int, expert_rows, expected_rows: int, atype, x,
                        ldx: int, y, ldy: int, workspace, ws_bytes: int, flags: int = 0, stream=None) -> None:
    _check(lib().hq_moe_grouped_gemm(ctypes.byref(desc), _ptr(w_t), form, rows, _ptr(expert_rows), expected_rows,
                                     ATYPES.get(atype, atype), _ptr(x), ldx, _ptr(y), ldy, _ptr(workspace),
                                     ws_bytes, flags, _stream(stream)), "hq_moe_grouped_gemm")


def hq_status_read(workspace, clear: bool = False, stream=None) -> int:
    out = ctypes.c_int32(0)
    _check(lib().hq_status_read(_ptr(workspace), 1 if clear else 0, _stream(stream), ctypes.byref(out)),
           "hq_status_read")
    return out.value


def _plan_dict(info: PlanInfo) -> dict:
    return {"bn": info.bn, "splits": info.splits, "grid": info.grid, "launches": info.launches,
            "stages": info.stages, "tile_class": info.tile_class, "groups": info.groups, "x_stages": info.x_stages}


def hq_selftest_wait_timeout(workspace, stream=None) -> None:
    _check(lib().hq_selftest_wait_timeout(_ptr(workspace), _stream(stream)), "hq_selftest_wait_timeout")


def hq_mxfp8_quantize(m: int, k: int, x, ldx: int, q, ldq: int, e, lde: int, stream=None) -> None:
    _check(lib().hq_mxfp8_quantize(m, k, _ptr(x), ldx, _ptr(q), ldq, _ptr(e), lde, _stream(stream)),
           "hq_mxfp8_quantize")


def hq_last_plan() -> dict:
    info = PlanInfo()
    _check(lib().hq_last_plan(ctypes.byref(info)), "hq_last_plan")
    return _plan_dict(info)


def hq_plan_query(desc: WeightDesc, m: int, atype, sms: int, smem_optin: int, flags: int = 0) -> dict:
    """The plan hq_gemm would choose on a device with `sms` SMs and `smem_optin`
    bytes of opt-in shared memory (host only: no device needed)."""
    info = PlanInfo()
    _check(lib().hq_plan_query(ctypes.byref(desc), m, ATYPES.get(atype, atype), sms, smem_optin, flags,
                               ctypes.byref(info)), "hq_plan_query")
    return _plan_dict(info)


def hq_moe_plan_query(desc: WeightDesc, tokens: int, topk: int, sms: int, smem_optin: int) -> dict:
    """The plan hq_moe_gemm would choose on such a device (host only)."""
    info = PlanInfo()
    _check(lib().hq_moe_plan_query(ctypes.byref(desc), tokens, topk, sms, smem_optin, ctypes.byref(info)),
           "hq_moe_plan_query")
    return _plan_dict(info)


def hq_tuning_reload() -> None:
    """Re-read the HQ_FORCE_* / HQ_TRACE switches from the environment."""
    lib().hq_tuning_reload()
