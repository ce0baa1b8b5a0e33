"""ctypes binding of libtpshard.so: one Python function per C entry point, same
name, same argument order.  Argument marshalling only -- every computation
runs in the library's CUDA kernels.

Tensor arguments may be torch tensors (their device pointer is passed), None
(NULL) or plain integers (raw device addresses).  ``stream=None`` means
torch's current CUDA stream.  A non-zero tp_status raises :class:`TPError`.
There is no fallback: if the library is not built, or no sm_103a GPU is
present, the calls fail loudly.
"""

from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtpshard.so")

TP_OK, TP_ERR_INVALID_ARG, TP_ERR_SHAPE, TP_ERR_ALIGN, TP_ERR_WORKSPACE, TP_ERR_CUDA, TP_ERR_TIMEOUT, \
    TP_ERR_UNSUPPORTED = range(8)
TP_ACT_IDENTITY, TP_ACT_RELU, TP_ACT_GELU_TANH, TP_ACT_GELU_ERF, TP_ACT_SWIGLU = range(5)
ACT_BY_NAME = {"identity": TP_ACT_IDENTITY, "relu": TP_ACT_RELU, "gelu_tanh": TP_ACT_GELU_TANH,
               "gelu_erf": TP_ACT_GELU_ERF, "swiglu": TP_ACT_SWIGLU}
TP_FLAG_UNFUSED_REDUCE = 1
TP_FLAG_OVERLAP_REDUCE = 2
TP_ATTN_F16_INPUT = 1

_P, _I64, _I, _U, _SZ, _F = C.c_void_p, C.c_int64, C.c_int, C.c_uint, C.c_size_t, C.c_float

# name -> (restype, [argtypes]); the last argument of every tp_status call is the stream.
SIGNATURES = {
    "tp_abi_version": (_I, []),
    "tp_status_string": (C.c_char_p, [_I]),
    "tp_get_device_status": (_I, [_P]),
    "tp_selftest_bounded_wait": (_I, [_I64, _P]),
    "tp_pack_col": (_I, [_P, _I64, _I64, _I, _P, _P]),
    "tp_unpack_col": (_I, [_P, _I64, _I64, _I, _P, _P]),
    "tp_pack_row": (_I, [_P, _I64, _I64, _I, _P, _P]),
    "tp_unpack_row": (_I, [_P, _I64, _I64, _I, _P, _P]),
    "tp_pack_swiglu": (_I, [_P, _P, _I64, _I64, _I, _P, _P]),
    "tp_pack_qkv_heads": (_I, [_P, _I64, _I, _I, _I, _P, _P]),
    "tp_unpack_qkv_heads": (_I, [_P, _I64, _I, _I, _I, _P, _P]),
    "tp_pack_qkv_bias": (_I, [_P, _I64, _I, _I, _I, _P, _P]),
    "tp_pack_qkv_gqa": (_I, [_P, _I64, _I, _I, _I, _I, _P, _P]),
    "tp_unpack_qkv_gqa": (_I, [_P, _I64, _I, _I, _I, _I, _P, _P]),
    "tp_pack_qkv_gqa_bias": (_I, [_P, _I, _I, _I, _I, _P, _P]),
    "tp_mlp_workspace_size": (_SZ, [_I64, _I64, _I64, _I, _U]),
    "tp_mlp_forward": (_I, [_P, _I64, _I64, _I64, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _U, _P, _SZ, _P]),
    "tp_mlp_backward_workspace_size": (_SZ, [_I64, _I64, _I64, _I, _U]),
    "tp_mlp_backward": (_I, [_P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _P, _P, _P, _P, _P, _P, _P, _I, _U, _P,
                             _SZ, _P]),
    "tp_kernel_launch_count": (C.c_uint64, []),
    "tp_last_error_detail": (C.c_char_p, []),
    "tp_column_parallel_forward": (_I, [_P, _I64, _I64, _I64, _I, _I, _P, _P, _P, _P, _P]),
    "tp_row_parallel_forward": (_I, [_P, _I64, _I64, _I64, _I, _P, _P, _P, _P, _P]),
    "tp_column_parallel_workspace_size": (_SZ, [_I64, _I64, _I64, _I]),
    "tp_column_parallel_forward_ws": (_I, [_P, _I64, _I64, _I64, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "tp_row_parallel_workspace_size": (_SZ, [_I64, _I64, _I64, _I]),
    "tp_row_parallel_forward_ws": (_I, [_P, _I64, _I64, _I64, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "tp_attn_forward_workspace_size": (_SZ, [_I64, _I64, _I, _I, _I, _U]),
    "tp_row_parallel_overlap_workspace_size": (_SZ, [_I64, _I64, _I64, _I]),
    "tp_row_parallel_forward_overlap": (_I, [_P, _I64, _I64, _I64, _I, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "tp_decode_swiglu_forward": (_I, [_P, _I64, _I64, _I64, _I, _P, _P, _P, _P, _P]),
    "tp_decode_attn_workspace_size": (_SZ, [_I64, _I64, _I, _I, _I, _I, _I64]),
    "tp_decode_attn_forward": (_I, [_P, _I64, _I64, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P, _I64, _P, _P, _P,
                                    _SZ, _P]),
    "tp_vocab_embedding_forward": (_I, [_P, _I64, _I64, _I64, _I, _P, _P, _P]),
    "tp_vocab_embedding_backward_workspace_size": (_SZ, [_I64]),
    "tp_vocab_embedding_backward": (_I, [_P, _P, _I64, _I64, _I64, _I, _P, _I, _P, _SZ, _P]),
    "tp_sp_layernorm_forward": (_I, [_P, _I64, _I64, _I, _P, _P, _F, _P, _P, _P, _P]),
    "tp_sp_layernorm_backward": (_I, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I, _P, _P, _P, _P, _P, _P]),
    "tp_sp_layernorm_forward_f16": (_I, [_P, _I64, _I64, _I, _P, _P, _F, _P, _P, _P, _P]),
    "tp_convert_bf16_to_f16": (_I, [_P, _I64, _P, _P]),
    "tp_attn_forward": (_I, [_P, _I64, _I64, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P, _P, _P, _P, _U, _P, _SZ,
                             _P]),
    "tp_attn_gqa_forward": (_I, [_P, _I64, _I64, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P, _P, _P, _P, _U,
                                 _P, _SZ, _P]),
    "tp_attn_gqa_backward_workspace_size": (_SZ, [_I64, _I64, _I, _I, _I, _I, _U]),
    "tp_attn_gqa_backward": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P,
                                  _P, _I, _U, _P, _SZ, _P]),
    "tp_reduce_qkv_gqa_grad": (_I, [_P, _I64, _I, _I, _I, _I, _P, _I, _P]),
    "tp_attn_core_forward": (_I, [_P, _I64, _I64, _I, _I, _I, _I, _I, _F, _P, _P, _P]),
    "tp_attn_core_backward": (_I, [_P, _P, _P, _P, _I64, _I64, _I, _I, _I, _I, _I, _F, _P, _P, _P]),
    "tp_attn_backward_workspace_size": (_SZ, [_I64, _I64, _I, _I, _I, _U]),
    "tp_attn_backward": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P, _P, _I, _U,
                              _P, _SZ, _P]),
    "tp_shard_reduce": (_I, [_P, _I64, _I64, _I, _P, _P, _P, _P, _P]),
    "tp_colsum_workspace_size": (_SZ, [_I64, _I64]),
    "tp_colsum": (_I, [_P, _I64, _I64, _P, _I, _P, _SZ, _P]),
    "tp_colsum_noalloc": (_I, [_P, _I64, _I64, _P, _I, _P]),
}


class TPError(RuntimeError):
    def __init__(self, name, status, message):
        super().__init__(f"{name} -> {message}")
        self.status = status


_lib = None


def lib():
    """The loaded library.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(python -m megatron_tensor_transformer_shard_gb300.build)")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if getattr(x, "is_cuda", True) is False:
            raise ValueError("tensor arguments must live on the GPU")
        return x.data_ptr()
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def status_string(code: int) -> str:
    return lib().tp_status_string(code).decode()


def _make(name):
    res, args = SIGNATURES[name]
    returns_status = res is _I and name not in ("tp_abi_version",)
    has_stream = bool(args) and name not in ("tp_status_string",) and returns_status

    def call(*a, stream=None, check=True):
        fn = getattr(lib(), name)
        n_user = len(args) - (1 if has_stream else 0)
        if len(a) != n_user:
            raise TypeError(f"{name} takes {n_user} arguments ({len(a)} given)")
        conv = []
        for v, ty in zip(a, args):
            conv.append(_ptr(v) if ty is _P else v)
        if has_stream:
            conv.append(_stream(stream))
        r = fn(*conv)
        if returns_status and check and r != TP_OK:
            msg = status_string(r)
            if r == TP_ERR_CUDA:
                msg += " [" + lib().tp_last_error_detail().decode() + "]"
            raise TPError(name, r, msg)
        return r

    call.__name__ = name
    call.__doc__ = f"Binding of the C entry point {name} (see include/tp.h)."
    return call


for _name in SIGNATURES:
    globals()[_name] = _make(_name)

__all__ = ["lib", "TPError", "status_string", "SIGNATURES", "LIB_PATH", "ACT_BY_NAME",
           "TP_FLAG_UNFUSED_REDUCE", "TP_FLAG_OVERLAP_REDUCE"] + list(SIGNATURES)
