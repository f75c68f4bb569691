"""ctypes binding of libnvfp4gemm.so: the C entry points under the same names,
argument marshalling only.  Every computation runs in the library's CUDA
kernels; there is no fallback path.

Pointer arguments accept either an integer device address or any object with
``data_ptr()`` (a torch tensor).  ``stream`` accepts None (torch's current
stream on the current device), an integer handle, or a ``torch.cuda.Stream``.
Errors raise ``Nvfp4Error`` carrying the status code and the library's message.
"""
import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libnvfp4gemm.so")
HEADER_PATH = os.path.join(os.path.dirname(HERE), "include", "nvfp4_gemm.h")

STATUS = {
    0: "NVFP4_OK",
    -1: "NVFP4_ERR_INVALID_ARG",
    -2: "NVFP4_ERR_UNSUPPORTED_SHAPE",
    -3: "NVFP4_ERR_CUDA",
    -4: "NVFP4_ERR_DEVICE_TIMEOUT",
    -5: "NVFP4_ERR_UNSUPPORTED_DEVICE",
}
MAX_GROUPS = 8


class Nvfp4Error(RuntimeError):
    def __init__(self, code, func, msg):
        super().__init__("%s -> %s: %s" % (func, STATUS.get(code, code), msg))
        self.code = code
        self.func = func


_lib = None


def load_library(path=LIB_PATH):
    """Load the shared library (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError("libnvfp4gemm.so is not built (%s); run __graft_entry__.build()" % path)
    lib = ctypes.CDLL(path)
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    vpp = ctypes.POINTER(ctypes.c_void_p)
    ip = ctypes.POINTER(ctypes.c_int)
    lib.nvfp4_gemm_repacked_scales_bytes.argtypes = [i, i, i]
    lib.nvfp4_gemm_repacked_scales_bytes.restype = sz
    lib.nvfp4_gemm_repack_scales.argtypes = [vp, vp, i, i, i, vp]
    lib.nvfp4_gemm_repack_scales.restype = i
    lib.nvfp4_gemm_run.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, vp]
    lib.nvfp4_gemm_run.restype = i
    lib.nvfp4_gemm_run_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, vp]
    lib.nvfp4_gemm_run_noalloc.restype = i
    lib.nvfp4_gemm_run_grouped.argtypes = [i, vpp, vpp, vpp, vpp, vpp, ip, ip, ip, ip, vp]
    lib.nvfp4_gemm_run_grouped.restype = i
    lib.nvfp4_gemm_last_error_string.argtypes = []
    lib.nvfp4_gemm_last_error_string.restype = ctypes.c_char_p
    lib.nvfp4_gemm_check_device_status.argtypes = [vp]
    lib.nvfp4_gemm_check_device_status.restype = i
    lib.nvfp4_gemm_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    lib.nvfp4_gemm_set_wait_timeout_ns.restype = i
    lib.nvfp4_gemm_debug_inject_skip.argtypes = [i]
    lib.nvfp4_gemm_debug_inject_skip.restype = i
    lib.nvfp4_gemm_plan.argtypes = [i, ip, ip, ip, ip, i, ip, i]
    lib.nvfp4_gemm_plan.restype = i
    lib.nvfp4_gemm_debug_schedule.argtypes = [i, ip, ip, ip, ip, i, i, ip, i]
    lib.nvfp4_gemm_debug_schedule.restype = i
    lib.nvfp4_quantize.argtypes = [vp, i, vp, vp, i, i, i, vp]
    lib.nvfp4_quantize.restype = i
    lib.nvfp4_gemm_last_launch.argtypes = [ip, i]
    lib.nvfp4_gemm_last_launch.restype = i
    lib.nvfp4_gemm_encode_idesc.argtypes = [i, i]
    lib.nvfp4_gemm_encode_idesc.restype = ctypes.c_uint32
    lib.nvfp4_gemm_encode_smem_desc.argtypes = [ctypes.c_uint32, i]
    lib.nvfp4_gemm_encode_smem_desc.restype = ctypes.c_uint64
    _lib = lib
    return lib


def header_functions(path=HEADER_PATH):
    """Names of the functions declared in include/nvfp4_gemm.h."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_\w+)\s*\(", text)))


def _ptr(x):
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return ctypes.c_void_p(x.data_ptr())
    return ctypes.c_void_p(int(x))


def _stream(s):
    if s is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if hasattr(s, "cuda_stream"):
        return ctypes.c_void_p(s.cuda_stream)
    return ctypes.c_void_p(int(s))


def _check(rc, func):
    if rc != 0:
        raise Nvfp4Error(rc, func, nvfp4_gemm_last_error_string())


# ------------------------------------------------------------------ entry points
def nvfp4_gemm_repacked_scales_bytes(rows, K, L=1):
    return int(load_library().nvfp4_gemm_repacked_scales_bytes(rows, K, L))


def nvfp4_gemm_repack_scales(sf, out, rows, K, L=1, stream=None):
    rc = load_library().nvfp4_gemm_repack_scales(_ptr(sf), _ptr(out), rows, K, L, _stream(stream))
    _check(rc, "nvfp4_gemm_repack_scales")


def nvfp4_gemm_run(A, B, SFA, SFB, C, M, N, K, L=1, stream=None):
    rc = load_library().nvfp4_gemm_run(_ptr(A), _ptr(B), _ptr(SFA), _ptr(SFB), _ptr(C), M, N, K, L,
                                       _stream(stream))
    _check(rc, "nvfp4_gemm_run")


def nvfp4_gemm_run_noalloc(A, B, SFA, SFB, C, M, N, K, L=1, stream=None):
    """nvfp4_gemm_run for callers that cannot allocate device memory: the
    split-K scratch is a static device array (see include/nvfp4_gemm.h)."""
    rc = load_library().nvfp4_gemm_run_noalloc(_ptr(A), _ptr(B), _ptr(SFA), _ptr(SFB), _ptr(C), M, N, K,
                                               L, _stream(stream))
    _check(rc, "nvfp4_gemm_run_noalloc")


DTYPE_BF16 = 0
DTYPE_F16 = 1


def nvfp4_quantize(x, x_dtype, codes, sf_repacked, rows, K, L=1, stream=None):
    rc = load_library().nvfp4_quantize(_ptr(x), int(x_dtype), _ptr(codes), _ptr(sf_repacked), rows, K, L,
                                       _stream(stream))
    _check(rc, "nvfp4_quantize")


def nvfp4_gemm_run_grouped(G, A, B, SFA, SFB, C, M, N, K, L, stream=None):
    def parr(xs):
        arr = (ctypes.c_void_p * max(G, 1))()
        for j in range(min(G, len(xs))):
            p = _ptr(xs[j])
            arr[j] = p.value if p is not None else None
        return arr

    def iarr(xs):
        arr = (ctypes.c_int * max(G, 1))()
        for j in range(min(G, len(xs))):
            arr[j] = int(xs[j])
        return arr

    rc = load_library().nvfp4_gemm_run_grouped(G, parr(A), parr(B), parr(SFA), parr(SFB), parr(C),
                                               iarr(M), iarr(N), iarr(K), iarr(L), _stream(stream))
    _check(rc, "nvfp4_gemm_run_grouped")


def nvfp4_gemm_last_error_string():
    return load_library().nvfp4_gemm_last_error_string().decode(errors="replace")


def nvfp4_gemm_check_device_status(stream=None):
    rc = load_library().nvfp4_gemm_check_device_status(_stream(stream))
    _check(rc, "nvfp4_gemm_check_device_status")


def nvfp4_gemm_set_wait_timeout_ns(ns):
    _check(load_library().nvfp4_gemm_set_wait_timeout_ns(int(ns)), "nvfp4_gemm_set_wait_timeout_ns")


def nvfp4_gemm_debug_inject_skip(ktile):
    _check(load_library().nvfp4_gemm_debug_inject_skip(int(ktile)), "nvfp4_gemm_debug_inject_skip")


def nvfp4_gemm_plan(M, N, K, L, num_sms):
    """Host-only launch plan (see include/nvfp4_gemm.h) as a dict."""
    G = len(M)
    ia = lambda xs: (ctypes.c_int * G)(*[int(v) for v in xs])
    out = (ctypes.c_int * 11)()
    rc = load_library().nvfp4_gemm_plan(G, ia(M), ia(N), ia(K), ia(L), num_sms, out, 11)
    _check(rc, "nvfp4_gemm_plan")
    keys = ("bn", "tiles", "grid", "stages", "dp_tiles", "sk_tiles", "sk_iters", "sk_max_segs", "cluster",
            "pair", "cluster_reduce")
    return dict(zip(keys, list(out)))


LAUNCH_VARIANTS = {-1: None, 0: "single", 1: "multicast", 2: "pair", 3: "cluster_reduce"}


def nvfp4_gemm_last_launch():
    """What this thread's last GEMM launch ran (see include/nvfp4_gemm.h)."""
    out = (ctypes.c_int * 5)()
    _check(load_library().nvfp4_gemm_last_launch(out, 5), "nvfp4_gemm_last_launch")
    return {"bn": out[0], "grid": out[1], "cluster": out[2], "variant": LAUNCH_VARIANTS.get(out[3], out[3]),
            "stages": out[4]}


def nvfp4_gemm_debug_schedule(M, N, K, L, num_sms, cta):
    """Host-only work list of one CTA: list of dicts (g, l, tm, tn, kt0, kt1,
    tile, seg, nseg)."""
    G = len(M)
    ia = lambda xs: (ctypes.c_int * G)(*[int(v) for v in xs])
    cap = 9 * 4096
    out = (ctypes.c_int * cap)()
    n = load_library().nvfp4_gemm_debug_schedule(G, ia(M), ia(N), ia(K), ia(L), num_sms, cta, out, cap)
    if n < 0:
        _check(n, "nvfp4_gemm_debug_schedule")
    keys = ("g", "l", "tm", "tn", "kt0", "kt1", "tile", "seg", "nseg")
    return [dict(zip(keys, out[9 * i:9 * i + 9])) for i in range(min(n, cap // 9))]


def nvfp4_gemm_encode_idesc(M, N):
    return int(load_library().nvfp4_gemm_encode_idesc(M, N))


def nvfp4_gemm_encode_smem_desc(addr, swizzle128):
    return int(load_library().nvfp4_gemm_encode_smem_desc(addr, 1 if swizzle128 else 0))


# ------------------------------------------------------------------ torch helpers
def repack_scales(sf, rows, K, L=1, stream=None):
    """Allocate the repacked buffer (torch, on sf's device) and fill it."""
    import torch
    out = torch.empty(nvfp4_gemm_repacked_scales_bytes(rows, K, L), dtype=torch.uint8, device=sf.device)
    nvfp4_gemm_repack_scales(sf, out, rows, K, L, stream)
    return out


def gemm(A, B, SFA_rp, SFB_rp, M, N, K, L=1, C=None, stream=None):
    """C [L, M, N] fp16 = A * SFA * B * SFB via nvfp4_gemm_run."""
    import torch
    if C is None:
        C = torch.empty((L, M, N), dtype=torch.float16, device=A.device)
    nvfp4_gemm_run(A, B, SFA_rp, SFB_rp, C, M, N, K, L, stream)
    return C


def quantize(x, stream=None):
    """x [L, rows, K] or [rows, K] bf16 / fp16 torch tensor on the GPU ->
    (codes [L, rows, K/2] u8, repacked scales u8) via nvfp4_quantize."""
    import torch
    if x.dim() == 2:
        x = x.unsqueeze(0)
    L, rows, K = x.shape
    dtype = {torch.bfloat16: DTYPE_BF16, torch.float16: DTYPE_F16}[x.dtype]
    x = x.contiguous()
    codes = torch.empty((L, rows, K // 2), dtype=torch.uint8, device=x.device)
    sf = torch.empty(nvfp4_gemm_repacked_scales_bytes(rows, K, L), dtype=torch.uint8, device=x.device)
    nvfp4_quantize(x, dtype, codes, sf, rows, K, L, stream)
    return codes, sf
