"""Python binding of libkvq: certified quantized-KV decode attention on GB300 (sm_103a).

Argument marshalling only: every step of the path runs in the CUDA kernels of
``libkvq.so`` behind the C ABI declared in ``include/kvq.h``.  Torch supplies device
memory and streams.  Importing this module fails loudly if the library is not built
(``python -c "import __graft_entry__ as g; g.build()"``); there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")

KVQ_OK = 0
KVQ_ERR_INVALID = 1
KVQ_ERR_OOM = 2
KVQ_ERR_HOST_OOM = 3
KVQ_ERR_CAPACITY = 4
KVQ_ERR_CUDA = 5
KVQ_ERR_TIMEOUT = 6

DEBUG_FORCE_RANK_FAIL = 0x1
DEBUG_FORCE_DENSE = 0x2
DEBUG_SYNC = 0x4
DEBUG_PROFILE = 0x8
DEBUG_BOUNDS = 0x10
DEBUG_FAIL_MIRROR = 0x20

HEAD_DIM = 128
BLOCK = 64
VALUE_GROUP = 32


class KvqError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"kvq status {status}: {msg}")
        self.status = status


class kvq_config(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int), ("batch", ctypes.c_int), ("n_q_heads", ctypes.c_int),
        ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("block_tokens", ctypes.c_int),
        ("value_group", ctypes.c_int), ("max_ctx", ctypes.c_int), ("rank_positions", ctypes.c_int),
        ("l4_head_fraction", ctypes.c_float), ("value_bits", ctypes.c_int),
        ("v_tol", ctypes.c_float), ("resident_blocks", ctypes.c_int),
    ]


class kvq_kernel_stat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int64), ("total_ms", ctypes.c_double)]


CERT_DTYPE = np.dtype([("e_key", "<f4"), ("e_val", "<f4"), ("rank_ok", "<i4"), ("level", "<i4"),
                       ("k_star", "<i4"), ("n_val_promoted", "<i4"), ("promoted_bytes", "<i8")])
assert CERT_DTYPE.itemsize == 32

_lib = None


def load_library() -> ctypes.CDLL:
    """Load libkvq.so from this package directory (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libkvq.so not built at {LIB_PATH}; run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    sigs = {
        "kvq_cache_create": [ctypes.POINTER(kvq_config), ctypes.POINTER(vp)],
        "kvq_cache_destroy": [vp],
        "kvq_append": [vp, i32, vp, vp, i32, vp],
        "kvq_decode_attention": [vp, i32, vp, f32, f32, vp, vp, vp, vp],
        "kvq_decode_attention_uncertified": [vp, i32, vp, vp, vp, vp],
        "kvq_set_debug": [vp, i32],
        "kvq_cache_length": [vp, i32, ctypes.POINTER(i32)],
        "kvq_export_tier1": [vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp],
        "kvq_export_decode_state": [vp, vp, vp, vp, vp, vp, vp, vp],
        "kvq_profile_read": [vp, ctypes.POINTER(kvq_kernel_stat), i32, ctypes.POINTER(i32), i32],
        "kvq_dense_decode_noalloc": [vp, vp, vp, i32, i32, i32, i32, vp, vp],
        "kvq_dense_attention_workspace": [i32, i32, i32, i32, ctypes.POINTER(ctypes.c_size_t)],
        "kvq_dense_attention": [vp, vp, vp, i32, i32, i32, i32, vp, vp, ctypes.c_size_t, vp],
        "kvq_debug_fill_tier2": [vp, i32, ctypes.c_uint16],
        "kvq_residency_stats": [vp, i32, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64),
                                ctypes.POINTER(i32), i32],
    }
    for name, argt in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = argt
        fn.restype = ctypes.c_int
    lib.kvq_last_error.argtypes = []
    lib.kvq_last_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(status: int):
    if status != KVQ_OK:
        raise KvqError(status, load_library().kvq_last_error().decode())


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _need(t, name, dtype, shape=None, nbytes=None):
    """Check a tensor argument before its pointer crosses the C ABI (which sees only the
    address): contiguous, of `dtype`, and of `shape` or `nbytes` when given."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if nbytes is not None and t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{name} must hold at least {nbytes} bytes")


def _stream(stream) -> int | None:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream or None
    return getattr(stream, "cuda_stream", stream) or None


def certificates(raw) -> np.ndarray:
    """View a raw certificate buffer (torch uint8 tensor or bytes) as a structured array."""
    import torch
    if isinstance(raw, torch.Tensor):
        raw = raw.detach().cpu().numpy()
    return np.frombuffer(np.ascontiguousarray(raw).tobytes(), dtype=CERT_DTYPE)


class Cache:
    """A tiered certified KV cache for `n_layers` layers (kvq_cache_create)."""

    def __init__(self, n_layers, batch, n_q_heads, n_kv_heads, max_ctx, rank_positions=1,
                 l4_head_fraction=0.5, head_dim=HEAD_DIM, block_tokens=BLOCK,
                 value_group=VALUE_GROUP, value_bits=4, v_tol=0.0, resident_blocks=0):
        self.lib = load_library()
        self.cfg = kvq_config(n_layers, batch, n_q_heads, n_kv_heads, head_dim, block_tokens,
                              value_group, max_ctx, rank_positions, l4_head_fraction, value_bits,
                              v_tol, resident_blocks)
        self.value_bits = value_bits
        h = ctypes.c_void_p()
        _check(self.lib.kvq_cache_create(ctypes.byref(self.cfg), ctypes.byref(h)))
        self.handle = h
        self.batch, self.n_q_heads, self.n_kv_heads = batch, n_q_heads, n_kv_heads

    def close(self):
        if getattr(self, "handle", None):
            self.lib.kvq_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_debug(self, flags: int):
        _check(self.lib.kvq_set_debug(self.handle, flags))

    def length(self, layer: int) -> int:
        n = ctypes.c_int()
        _check(self.lib.kvq_cache_length(self.handle, layer, ctypes.byref(n)))
        return n.value

    def append(self, layer: int, k, v, stream=None):
        """k, v: contiguous fp16 CUDA tensors [B, Hkv, n, 128]."""
        import torch
        if k.dim() != 4:
            raise ValueError("k must be [batch, n_kv_heads, n_tokens, 128]")
        shape = (self.batch, self.n_kv_heads, k.shape[2], HEAD_DIM)
        _need(k, "k", torch.float16, shape)
        _need(v, "v", torch.float16, shape)
        _check(self.lib.kvq_append(self.handle, layer, _ptr(k), _ptr(v), k.shape[2], _stream(stream)))

    def decode(self, layer: int, q, tau_cov: float, eps: float, out, cert=None, ladder_level=None,
               stream=None):
        """q, out: contiguous fp16 tensors [B, Hq, 128] (device or host); cert: uint8 tensor
        of B*Hq*32 bytes or None; ladder_level: int32 tensor [B] or None.  Pinned host
        tensors are copied in stream order (read the results after a synchronize);
        pageable host tensors make the call wait for its copies."""
        self._check_decode_args(q, out, cert)
        if ladder_level is not None:
            import torch
            _need(ladder_level, "ladder_level", torch.int32, (self.batch,))
        st = _stream(stream) if (q.is_cuda or out.is_cuda) else None
        _check(self.lib.kvq_decode_attention(self.handle, layer, _ptr(q), float(tau_cov), float(eps),
                                             _ptr(out), _ptr(cert), _ptr(ladder_level), st))

    def decode_uncertified(self, layer: int, q, out, cert=None, stream=None):
        """Plain INT8/INT4 decode attention, nothing paged in and no ladder
        (kvq_decode_attention_uncertified); cert receives the unenforced bounds."""
        self._check_decode_args(q, out, cert)
        st = _stream(stream) if (q.is_cuda or out.is_cuda) else None
        _check(self.lib.kvq_decode_attention_uncertified(self.handle, layer, _ptr(q), _ptr(out),
                                                         _ptr(cert), st))

    def _check_decode_args(self, q, out, cert):
        import torch
        shape = (self.batch, self.n_q_heads, HEAD_DIM)
        _need(q, "q", torch.float16, shape)
        _need(out, "out", torch.float16, shape)
        if cert is not None:
            _need(cert, "cert", torch.uint8, nbytes=self.batch * self.n_q_heads * CERT_DTYPE.itemsize)

    def export_tier1(self, layer: int, stream=None) -> dict:
        """Tier-1 contents of `layer` in canonical layout, as CUDA tensors."""
        import torch
        B, H, n = self.batch, self.n_kv_heads, self.length(layer)
        nb = n // BLOCK
        dev = torch.device("cuda")
        out = dict(
            kc=torch.empty(B, H, nb, BLOCK, HEAD_DIM, dtype=torch.int8, device=dev),
            ks=torch.empty(B, H, nb, HEAD_DIM, dtype=torch.float16, device=dev),
            vc=torch.empty(B, H, nb, BLOCK, HEAD_DIM, dtype=torch.uint8, device=dev),
            vs=torch.empty(B, H, nb, BLOCK, HEAD_DIM // VALUE_GROUP, dtype=torch.float16, device=dev),
            vo=torch.empty(B, H, nb, BLOCK, HEAD_DIM // VALUE_GROUP, dtype=torch.float16, device=dev),
            eta=torch.empty(B, H, nb, dtype=torch.float32, device=dev),
            vmin=torch.empty(B, H, HEAD_DIM, dtype=torch.float32, device=dev),
            vmax=torch.empty(B, H, HEAD_DIM, dtype=torch.float32, device=dev),
        )
        o = out
        _check(self.lib.kvq_export_tier1(self.handle, layer, _ptr(o["kc"]), _ptr(o["ks"]), _ptr(o["vc"]),
                                         _ptr(o["vs"]), _ptr(o["vo"]), _ptr(o["eta"]), _ptr(o["vmin"]),
                                         _ptr(o["vmax"]), _stream(stream)))
        return out

    def export_decode_state(self, nb: int, stream=None) -> dict:
        """Selection state of the last certified decode call (nb = its full blocks)."""
        import torch
        B, Hq, H = self.batch, self.n_q_heads, self.n_kv_heads
        dev = torch.device("cuda")
        o = dict(
            sel=torch.zeros(B, Hq, nb, dtype=torch.uint8, device=dev),
            kprom0=torch.zeros(B, H, nb, dtype=torch.uint8, device=dev),
            kprom1=torch.zeros(B, H, nb, dtype=torch.uint8, device=dev),
            vprom1=torch.zeros(B, H, nb, dtype=torch.uint8, device=dev),
            lse8=torch.zeros(B, Hq, nb, dtype=torch.float32, device=dev),
            delta=torch.zeros(B, Hq, nb, dtype=torch.float32, device=dev),
        )
        _check(self.lib.kvq_export_decode_state(self.handle, _ptr(o["sel"]), _ptr(o["kprom0"]),
                                                _ptr(o["kprom1"]), _ptr(o["vprom1"]), _ptr(o["lse8"]),
                                                _ptr(o["delta"]), _stream(stream)))
        return o

    def residency_stats(self, layer: int, reset: bool = False) -> dict:
        """FP16 block bytes of `layer` served from resident HBM copies and read over the
        host link since the last reset, and the slots in use (kvq_residency_stats)."""
        hit, host, used = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int()
        _check(self.lib.kvq_residency_stats(self.handle, layer, ctypes.byref(hit), ctypes.byref(host),
                                            ctypes.byref(used), int(reset)))
        return {"resident_bytes": hit.value, "host_bytes": host.value, "slots_in_use": used.value}

    def debug_fill_tier2(self, layer: int, bits: int):
        """Test aid (kvq_debug_fill_tier2): overwrite `layer`'s tier-2 FP16 originals with
        the binary16 bit pattern `bits`, after the device has finished queued work."""
        _check(self.lib.kvq_debug_fill_tier2(self.handle, layer, int(bits) & 0xFFFF))

    def profile_read(self, reset: bool = True) -> dict:
        arr = (kvq_kernel_stat * 16)()
        n = ctypes.c_int()
        _check(self.lib.kvq_profile_read(self.handle, arr, 16, ctypes.byref(n), int(reset)))
        return {arr[i].name.decode(): (arr[i].launches, arr[i].total_ms) for i in range(n.value)}


def dense_decode_noalloc(q, k, v, out, stream=None):
    """Exact dense FP16 decode attention with no allocation (kvq_dense_decode_noalloc).

    For callers that cannot allocate device memory at call time; q, out: device fp16
    [B, Hq, 128]; k, v: device fp16 [B, Hkv, n_tokens, 128].  Its scratch is a fixed
    8 MiB device array shared by every call, so overlapping calls must be serialised.
    """
    import torch
    if q.dim() != 3 or k.dim() != 4:
        raise ValueError("q must be [batch, n_q_heads, 128] and k, v [batch, n_kv_heads, n_tokens, 128]")
    B, Hq, _ = q.shape
    Hkv, N = k.shape[1], k.shape[2]
    _need(q, "q", torch.float16, (B, Hq, HEAD_DIM))
    _need(k, "k", torch.float16, (B, Hkv, N, HEAD_DIM))
    _need(v, "v", torch.float16, (B, Hkv, N, HEAD_DIM))
    _need(out, "out", torch.float16, (B, Hq, HEAD_DIM))
    dev = q.device
    if any(t.device != dev for t in (k, v, out)):
        raise ValueError("q, k, v and out must be on one CUDA device")
    if dev.type == "cuda":
        with torch.cuda.device(dev):   # the call runs on the tensors' device and its stream
            _check(load_library().kvq_dense_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, N,
                                                           _ptr(out), _stream(stream)))
        return
    _check(load_library().kvq_dense_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, N,
                                                   _ptr(out), _stream(stream)))


def dense_attention_workspace(batch: int, n_q_heads: int, n_kv_heads: int, n_tokens: int) -> int:
    """Workspace bytes kvq_dense_attention needs for this shape on the current device."""
    n = ctypes.c_size_t(0)
    _check(load_library().kvq_dense_attention_workspace(batch, n_q_heads, n_kv_heads, n_tokens, ctypes.byref(n)))
    return int(n.value)


def dense_attention(q, k, v, out, workspace=None, stream=None):
    """Exact dense FP16 decode attention over K/V in device memory (kvq_dense_attention).

    q, out: device fp16 [B, Hq, 128]; k, v: device fp16 [B, Hkv, n_tokens, 128].
    `workspace` is a device uint8 tensor of at least dense_attention_workspace(...) bytes
    (allocated here when omitted).  Returns `workspace` so a caller can reuse it.
    """
    import torch
    if q.dim() != 3 or k.dim() != 4:
        raise ValueError("q must be [batch, n_q_heads, 128] and k, v [batch, n_kv_heads, n_tokens, 128]")
    B, Hq, _ = q.shape
    Hkv, N = k.shape[1], k.shape[2]
    _need(q, "q", torch.float16, (B, Hq, HEAD_DIM))
    _need(k, "k", torch.float16, (B, Hkv, N, HEAD_DIM))
    _need(v, "v", torch.float16, (B, Hkv, N, HEAD_DIM))
    _need(out, "out", torch.float16, (B, Hq, HEAD_DIM))
    dev = q.device
    if dev.type != "cuda" or any(t.device != dev for t in (k, v, out)):
        raise ValueError("q, k, v and out must be on one CUDA device")
    with torch.cuda.device(dev):
        need = dense_attention_workspace(B, Hq, Hkv, N)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        _need(workspace, "workspace", torch.uint8, nbytes=need)
        _check(load_library().kvq_dense_attention(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, N, _ptr(out),
                                                  _ptr(workspace), workspace.numel(), _stream(stream)))
    return workspace


def header_functions(header_path: str | None = None) -> list[str]:
    """Names of the functions declared in include/kvq.h."""
    import re
    path = header_path or os.path.join(os.path.dirname(_HERE), "include", "kvq.h")
    text = open(path).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_]+\s*\*?\s*(kvq_[a-z0-9_]+)\s*\(", text, re.M)))
