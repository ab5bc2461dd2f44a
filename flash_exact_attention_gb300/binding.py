"""ctypes binding of libattn.so (the C ABI in include/attn.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  PyTorch supplies device memory and the stream.
There is no fallback: if the library was not built, every call raises.
"""
import ctypes
import math
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_DEVICE_TIMEOUT = 4
ATTN_ERR_ARCH = 5
ATTN_ERR_SCRATCH_LIMIT = 6

_lib = None

# (name, argtypes, restype) for every function include/attn.h declares.
_P, _I, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
SIGNATURES = {
    "attn_fwd": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P], _I),
    "attn_bwd": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P], _I),
    "attn_bwd_noalloc": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P],
                         _I),
    "attn_fwd_f16": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P], _I),
    "attn_stieltjes_fwd": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P], _I),
    "attn_fwd_varlen": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P], _I),
    "attn_bwd_varlen": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P,
                         _P], _I),
    "attn_fwd_varlen_f16": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P], _I),
    "attn_bwd_varlen_f16": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P,
                             _P, _P], _I),
    "attn_nystrom_fwd": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _F, _P], _I),
    "attn_bwd_deterministic": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P,
                                _P], _I),
    "attn_bwd_f16": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P], _I),
    "attn_bwd_noalloc_scratch_limit": ([], ctypes.c_longlong),
    "attn_status_string": ([_I], ctypes.c_char_p),
    "attn_device_status": ([_P], _I),
    "attn_set_wait_timeout_ms": ([_I], _I),
    "attn_selftest_wait_timeout": ([_I, _P], _I),
    "attn_version": ([], _I),
}


class AttnError(RuntimeError):
    """A non-OK status from the C ABI."""

    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, status_text(status), status))


def load():
    """Loads libattn.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libattn.so is missing; build it with "
                               "`python -m flash_exact_attention_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def status_text(status):
    return load().attn_status_string(int(status)).decode()


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# --------------------------------------------------------------- raw C names
def attn_fwd(q, k, v, o, lse, B, Hq, Hkv, N, D, causal, scale, stream=None):
    """Raw call: pointers (ints) or tensors; returns the status code."""
    return load().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, D,
                           int(bool(causal)), float(scale), _stream_handle(stream))


def attn_bwd(q, k, v, o, lse, B, Hq, Hkv, N, D, causal, scale, stream, dout, dq, dk, dv):
    """Raw call: pointers (ints) or tensors; returns the status code."""
    return load().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, D,
                           int(bool(causal)), float(scale), _stream_handle(stream),
                           _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv))


def attn_fwd_f16(q, k, v, o, lse, B, Hq, Hkv, N, D, causal, scale, stream=None):
    """Raw call, fp16 tensors: pointers (ints) or tensors; returns the status code."""
    return load().attn_fwd_f16(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, D,
                               int(bool(causal)), float(scale), _stream_handle(stream))


def attn_bwd_f16(q, k, v, o, lse, B, Hq, Hkv, N, D, causal, scale, stream, dout, dq, dk, dv):
    """Raw call, fp16 tensors: pointers (ints) or tensors; returns the status code."""
    return load().attn_bwd_f16(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, D,
                               int(bool(causal)), float(scale), _stream_handle(stream),
                               _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv))


def attn_stieltjes_fwd(q, k, v, o, pole, B, Hq, Hkv, N, D, causal, scale, order, newton_steps,
                       stream=None):
    """Raw call of the Stieltjes attention forward; returns the status code."""
    return load().attn_stieltjes_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(pole), B, Hq, Hkv,
                                     N, D, int(bool(causal)), float(scale), int(order),
                                     int(newton_steps), _stream_handle(stream))


def attn_fwd_varlen(q, k, v, o, lse, cu_seqlens, B, Hq, Hkv, total, max_seqlen, D, causal, scale,
                    stream=None):
    """Raw call of the packed variable-length forward; returns the status code."""
    return load().attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens),
                                  B, Hq, Hkv, total, max_seqlen, D, int(bool(causal)),
                                  float(scale), _stream_handle(stream))


def attn_bwd_varlen(q, k, v, o, lse, cu_seqlens, B, Hq, Hkv, total, max_seqlen, D, causal, scale,
                    stream, dout, dq, dk, dv):
    """Raw call of the packed variable-length backward; returns the status code."""
    return load().attn_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens),
                                  B, Hq, Hkv, total, max_seqlen, D, int(bool(causal)),
                                  float(scale), _stream_handle(stream), _ptr(dout), _ptr(dq),
                                  _ptr(dk), _ptr(dv))


def attn_fwd_varlen_f16(q, k, v, o, lse, cu_seqlens, B, Hq, Hkv, total, max_seqlen, D, causal,
                        scale, stream=None):
    """Raw call of the fp16 packed variable-length forward; returns the status code."""
    return load().attn_fwd_varlen_f16(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                      _ptr(cu_seqlens), B, Hq, Hkv, total, max_seqlen, D,
                                      int(bool(causal)), float(scale), _stream_handle(stream))


def attn_bwd_varlen_f16(q, k, v, o, lse, cu_seqlens, B, Hq, Hkv, total, max_seqlen, D, causal,
                        scale, stream, dout, dq, dk, dv):
    """Raw call of the fp16 packed variable-length backward; returns the status code."""
    return load().attn_bwd_varlen_f16(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                      _ptr(cu_seqlens), B, Hq, Hkv, total, max_seqlen, D,
                                      int(bool(causal)), float(scale), _stream_handle(stream),
                                      _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv))


def attn_nystrom_fwd(q, k, v, o, B, Hq, Hkv, N, D, num_landmarks, newton_iters, kappa, scale,
                     stream=None):
    """Raw call of the Nystrom attention forward; returns the status code."""
    return load().attn_nystrom_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, Hq, Hkv, N, D,
                                   int(num_landmarks), int(newton_iters), float(kappa),
                                   float(scale), _stream_handle(stream))


def attn_bwd_deterministic(q, k, v, o, lse, B, Hq, Hkv, N, D, causal, scale, stream, dout, dq,
                           dk, dv):
    """Raw call of the run-to-run bitwise-reproducible backward (bf16)."""
    return load().attn_bwd_deterministic(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq,
                                         Hkv, N, D, int(bool(causal)), float(scale),
                                         _stream_handle(stream), _ptr(dout), _ptr(dq), _ptr(dk),
                                         _ptr(dv))


def attn_bwd_noalloc(q, k, v, o, lse, B, Hq, Hkv, N, D, causal, scale, stream, dout, dq, dk,
                     dv):
    """Raw call of the backward that allocates nothing (fixed scratch array)."""
    return load().attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N,
                                   D, int(bool(causal)), float(scale), _stream_handle(stream),
                                   _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv))


def attn_status_string(status):
    return status_text(status)


def attn_device_status(stream=None):
    return load().attn_device_status(_stream_handle(stream))


def attn_selftest_wait_timeout(timeout_ms, stream=None):
    """Enqueues a kernel whose bounded wait is made to run out (diagnostic)."""
    return load().attn_selftest_wait_timeout(int(timeout_ms), _stream_handle(stream))


def attn_set_wait_timeout_ms(ms):
    return load().attn_set_wait_timeout_ms(int(ms))


# ------------------------------------------------------- tensor conveniences
def _check(t, shape, name, dtype=None):
    import torch
    if dtype is None:
        dtype = t.dtype
    if dtype not in (torch.bfloat16, torch.float16) or t.dtype != dtype or not t.is_cuda or \
            not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA tensor of q's dtype (bf16 or fp16)" % name)
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))


def flash_attn(q, k, v, causal=False, scale=None, stream=None):
    """O, LSE = attention(q, k, v); q [B,Hq,N,D], k/v [B,Hkv,N,D] bf16 or fp16 on CUDA."""
    import torch
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    _check(q, (B, Hq, N, D), "q")
    _check(k, (B, Hkv, N, D), "k", q.dtype)
    _check(v, (B, Hkv, N, D), "v", q.dtype)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    call = attn_fwd_f16 if q.dtype == torch.float16 else attn_fwd
    st = call(q, k, v, o, lse, B, Hq, Hkv, N, D, causal, scale, stream)
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd")
    return o, lse


def flash_attn_bwd(q, k, v, o, lse, dout, causal=False, scale=None, stream=None,
                   deterministic=False):
    """dQ, dK, dV of sum(dout * O) given the forward's O and LSE.  With
    deterministic=True (bf16 only) the results are bitwise reproducible."""
    import torch
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    for t, shp, nm in ((q, (B, Hq, N, D), "q"), (k, (B, Hkv, N, D), "k"),
                       (v, (B, Hkv, N, D), "v"), (o, (B, Hq, N, D), "o"),
                       (dout, (B, Hq, N, D), "dout")):
        _check(t, shp, nm, q.dtype)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    if deterministic:
        if q.dtype != torch.bfloat16:
            raise ValueError("the deterministic backward takes bf16 tensors")
        call = attn_bwd_deterministic
    else:
        call = attn_bwd_f16 if q.dtype == torch.float16 else attn_bwd
    st = call(q, k, v, o, lse, B, Hq, Hkv, N, D, causal, scale, stream, dout, dq, dk, dv)
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd")
    return dq, dk, dv


_ATTN_FUNCTION = None


def _attn_function():
    """torch.autograd.Function over attn_fwd / attn_bwd (built on first use so
    that importing this module does not import torch)."""
    global _ATTN_FUNCTION
    if _ATTN_FUNCTION is None:
        import torch

        class AttnFunction(torch.autograd.Function):
            @staticmethod
            def forward(ctx, q, k, v, causal, scale):
                o, lse = flash_attn(q, k, v, causal=causal, scale=scale)
                ctx.save_for_backward(q, k, v, o, lse)
                ctx.causal, ctx.scale = causal, scale
                ctx.mark_non_differentiable(lse)
                return o, lse

            @staticmethod
            def backward(ctx, dout, dlse):
                q, k, v, o, lse = ctx.saved_tensors
                dq, dk, dv = flash_attn_bwd(q, k, v, o, lse, dout.contiguous(),
                                            causal=ctx.causal, scale=ctx.scale)
                return dq, dk, dv, None, None

        _ATTN_FUNCTION = AttnFunction
    return _ATTN_FUNCTION


def attention(q, k, v, causal=False, scale=None):
    """Differentiable O = softmax(scale q k^T) v for bf16 or fp16 CUDA tensors q [B,Hq,N,D],
    k/v [B,Hkv,N,D]: the forward is attn_fwd, the gradient attn_bwd (on torch's
    current stream).  Returns O; the row log-sum-exp is kept for the backward."""
    o, _ = _attn_function().apply(q, k, v, bool(causal),
                                  1.0 / math.sqrt(q.shape[-1]) if scale is None else scale)
    return o


_OPS_REGISTERED = False


def register_ops():
    """Registers torch.ops.flash_exact_attention.fwd / .bwd (torch.library
    custom ops over attn_fwd / attn_bwd, with shape-only fake implementations
    and the backward as their autograd formula), so that torch.compile can
    keep a call inside one graph.  Idempotent; returns the op namespace."""
    global _OPS_REGISTERED
    import torch
    if not _OPS_REGISTERED:
        @torch.library.custom_op("flash_exact_attention::fwd", mutates_args=())
        def _fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool,
                 scale: float) -> tuple[torch.Tensor, torch.Tensor]:
            return flash_attn(q, k, v, causal=causal, scale=scale)

        @_fwd.register_fake
        def _(q, k, v, causal, scale):
            B, Hq, N, _ = q.shape
            return torch.empty_like(q), q.new_empty((B, Hq, N), dtype=torch.float32)

        @torch.library.custom_op("flash_exact_attention::bwd", mutates_args=())
        def _bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                 lse: torch.Tensor, dout: torch.Tensor, causal: bool,
                 scale: float) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
            return flash_attn_bwd(q, k, v, o, lse, dout.contiguous(), causal=causal, scale=scale)

        @_bwd.register_fake
        def _(q, k, v, o, lse, dout, causal, scale):
            return torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

        def _setup(ctx, inputs, output):
            q, k, v, causal, scale = inputs
            o, lse = output
            ctx.save_for_backward(q, k, v, o, lse)
            ctx.causal, ctx.scale = causal, scale

        def _backward(ctx, dout, dlse):
            q, k, v, o, lse = ctx.saved_tensors
            dq, dk, dv = torch.ops.flash_exact_attention.bwd(q, k, v, o, lse, dout, ctx.causal,
                                                             ctx.scale)
            return dq, dk, dv, None, None

        _fwd.register_autograd(_backward, setup_context=_setup)
        _OPS_REGISTERED = True
    return torch.ops.flash_exact_attention


def attention_op(q, k, v, causal=False, scale=None):
    """attention() through the registered custom ops.  Inside torch.compile,
    call register_ops() once beforehand (registration itself is not traceable)."""
    import torch
    if not _OPS_REGISTERED:
        register_ops()
    o, _ = torch.ops.flash_exact_attention.fwd(
        q, k, v, bool(causal), 1.0 / math.sqrt(q.shape[-1]) if scale is None else float(scale))
    return o


def stieltjes_attn(q, k, v, causal=False, scale=None, order=4, newton_steps=3, stream=None):
    """Stieltjes attention (FlashStieltjes page): O and the per-row pole for bf16
    CUDA tensors q [B,Hq,N,D], k/v [B,Hkv,N,D]; order 2 or 4, newton_steps Newton
    steps from 1.1 above the row max (the page's default is 3)."""
    import torch
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    _check(q, (B, Hq, N, D), "q", torch.bfloat16)
    _check(k, (B, Hkv, N, D), "k", torch.bfloat16)
    _check(v, (B, Hkv, N, D), "v", torch.bfloat16)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = torch.empty_like(q)
    pole = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    st = attn_stieltjes_fwd(q, k, v, o, pole, B, Hq, Hkv, N, D, causal, scale, order,
                            newton_steps, stream)
    if st != ATTN_OK:
        raise AttnError(st, "attn_stieltjes_fwd")
    return o, pole


def nystrom_attn(q, k, v, num_landmarks=64, newton_iters=6, kappa=5.0, scale=None, stream=None):
    """Nystrom attention (FlashNystrom page) for bf16 CUDA tensors q [B,Hq,N,D],
    k/v [B,Hkv,N,D]: segment-mean landmarks, Newton-Schulz pseudo-inverse with
    the Tikhonov ridge kappa (0 = none).  The defaults are the page's
    (64 landmarks, 6 iterations, kappa 5)."""
    import torch
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    _check(q, (B, Hq, N, D), "q", torch.bfloat16)
    _check(k, (B, Hkv, N, D), "k", torch.bfloat16)
    _check(v, (B, Hkv, N, D), "v", torch.bfloat16)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = torch.empty_like(q)
    st = attn_nystrom_fwd(q, k, v, o, B, Hq, Hkv, N, D, num_landmarks, newton_iters, kappa,
                          scale, stream)
    if st != ATTN_OK:
        raise AttnError(st, "attn_nystrom_fwd")
    return o


def flash_attn_varlen(q, k, v, cu_seqlens, max_seqlen, causal=False, scale=None, stream=None):
    """O [total, Hq, D] and LSE [Hq, total] for sequences packed token-major:
    q [total, Hq, D], k/v [total, Hkv, D] bf16 or fp16 on CUDA; cu_seqlens an int32
    CUDA tensor [B + 1] of sequence offsets; max_seqlen at least the longest one."""
    import torch
    total, Hq, D = q.shape
    Hkv = k.shape[1]
    _check(q, (total, Hq, D), "q")
    _check(k, (total, Hkv, D), "k", q.dtype)
    _check(v, (total, Hkv, D), "v", q.dtype)
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor")
    B = cu_seqlens.numel() - 1
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = torch.empty_like(q)
    lse = torch.empty((Hq, total), dtype=torch.float32, device=q.device)
    call = attn_fwd_varlen_f16 if q.dtype == torch.float16 else attn_fwd_varlen
    st = call(q, k, v, o, lse, cu_seqlens.contiguous(), B, Hq, Hkv, total, int(max_seqlen), D,
              causal, scale, stream)
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_varlen")
    return o, lse


def flash_attn_varlen_bwd(q, k, v, o, lse, dout, cu_seqlens, max_seqlen, causal=False, scale=None,
                          stream=None):
    """dQ [total, Hq, D], dK, dV [total, Hkv, D] of sum(dout * O) for the packed
    batch flash_attn_varlen computed O [total, Hq, D] and LSE [Hq, total] of."""
    import torch
    total, Hq, D = q.shape
    Hkv = k.shape[1]
    for t, shp, nm in ((q, (total, Hq, D), "q"), (k, (total, Hkv, D), "k"),
                       (v, (total, Hkv, D), "v"), (o, (total, Hq, D), "o"),
                       (dout, (total, Hq, D), "dout")):
        _check(t, shp, nm, q.dtype)
    if (lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous()
            or tuple(lse.shape) != (Hq, total)):
        raise ValueError("lse must be a contiguous fp32 CUDA tensor [Hq, total]")
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor")
    B = cu_seqlens.numel() - 1
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    call = attn_bwd_varlen_f16 if q.dtype == torch.float16 else attn_bwd_varlen
    st = call(q, k, v, o, lse, cu_seqlens.contiguous(), B, Hq, Hkv, total, int(max_seqlen), D,
              causal, scale, stream, dout, dq, dk, dv)
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd_varlen")
    return dq, dk, dv


_VARLEN_FUNCTION = None


def _varlen_function():
    """torch.autograd.Function over attn_fwd_varlen / attn_bwd_varlen."""
    global _VARLEN_FUNCTION
    if _VARLEN_FUNCTION is None:
        import torch

        class VarlenAttnFunction(torch.autograd.Function):
            @staticmethod
            def forward(ctx, q, k, v, cu_seqlens, max_seqlen, causal, scale):
                o, lse = flash_attn_varlen(q, k, v, cu_seqlens, max_seqlen, causal=causal,
                                           scale=scale)
                ctx.save_for_backward(q, k, v, o, lse, cu_seqlens)
                ctx.max_seqlen, ctx.causal, ctx.scale = max_seqlen, causal, scale
                ctx.mark_non_differentiable(lse)
                return o, lse

            @staticmethod
            def backward(ctx, dout, dlse):
                q, k, v, o, lse, cu = ctx.saved_tensors
                dq, dk, dv = flash_attn_varlen_bwd(q, k, v, o, lse, dout.contiguous(), cu,
                                                   ctx.max_seqlen, causal=ctx.causal,
                                                   scale=ctx.scale)
                return dq, dk, dv, None, None, None, None

        _VARLEN_FUNCTION = VarlenAttnFunction
    return _VARLEN_FUNCTION


def attention_varlen(q, k, v, cu_seqlens, max_seqlen, causal=False, scale=None):
    """Differentiable attention over a packed batch of sequences of different
    lengths (layouts of flash_attn_varlen): the forward is attn_fwd_varlen, the
    gradient attn_bwd_varlen.  Returns O [total, Hq, D]."""
    o, _ = _varlen_function().apply(q, k, v, cu_seqlens, int(max_seqlen), bool(causal),
                                    1.0 / math.sqrt(q.shape[-1]) if scale is None else scale)
    return o
