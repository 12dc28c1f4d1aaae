"""Thin ctypes binding of libpkv.so (declared in include/pkv.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors; the stream defaults to torch's
current stream.  If the library has not been built, the first call raises --
there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpkv.so")

PKV_F32, PKV_BF16, PKV_FP8_E4M3 = 0, 1, 2
ALGOS = {"auto": 0, "simt": 1, "mma": 2, "tc": 3}
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "workspace", 4: "cuda error",
          5: "device bounds", 6: "out of blocks", 7: "inconsistent"}
ERRBIT_BLOCK_ID, ERRBIT_SLOT, ERRBIT_SEQ_LEN, ERRBIT_TIMEOUT = 1, 2, 4, 8

# Every symbol include/pkv.h declares.
EXPORTS = ("kv_pool_create", "kv_pool_destroy", "kv_pool_tensor_bytes", "kv_bytes_per_token",
           "kv_append", "paged_decode_plan", "paged_decode_algo", "paged_decode_attention",
           "paged_multi_query_plan", "paged_multi_query_algo", "paged_multi_query_attention",
           "paged_decode_append_attention",
           "paged_decode_attention_static_ws", "pkv_set_first_wait_limit_for_testing", "pkv_status_string",
           "pkv_last_cuda_error",
           "kv_block_manager_create", "kv_block_manager_destroy", "kv_bm_num_free", "kv_bm_add_sequence",
           "kv_bm_free_sequence", "kv_bm_grow", "kv_bm_decode_slots", "kv_bm_match_prefix", "kv_bm_seq_len",
           "kv_bm_block_tables", "kv_bm_free_list", "kv_bm_block_ref", "kv_bm_check")
STATIC_SCRATCH_BYTES = 16 * 1024 * 1024
ALGO_NAMES = {1: "simt", 2: "mma", 3: "tc"}


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = "%s failed: %s" % (what, STATUS.get(status, str(status)))
        if status == 4 and _lib is not None:
            msg += " (%s)" % _lib.pkv_last_cuda_error().decode()
        super().__init__(msg)


class PoolDesc(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("kv_dtype", ctypes.c_int), ("k_scale", ctypes.c_float),
                ("v_scale", ctypes.c_float), ("k_base", ctypes.c_void_p), ("v_base", ctypes.c_void_p),
                ("error_word", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libpkv.so (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libpkv.so is not built (run __graft_entry__.build() or "
                           "python -m paged_kv_cache_194_gb300.build); no fallback exists")
    L = ctypes.CDLL(LIB_PATH)
    c, P = ctypes, ctypes.c_void_p
    L.kv_pool_create.restype = c.c_int
    L.kv_pool_create.argtypes = [c.POINTER(PoolDesc), c.POINTER(P)]
    L.kv_pool_destroy.restype = None
    L.kv_pool_destroy.argtypes = [P]
    L.kv_pool_tensor_bytes.restype = c.c_size_t
    L.kv_pool_tensor_bytes.argtypes = [c.POINTER(PoolDesc)]
    L.kv_bytes_per_token.restype = c.c_int64
    L.kv_bytes_per_token.argtypes = [c.c_int32, c.c_int32, c.c_int32, c.c_int]
    L.kv_append.restype = c.c_int
    L.kv_append.argtypes = [P, c.c_int32, P, P, c.c_int, P, c.c_int32, P]
    L.paged_decode_plan.restype = c.c_int
    L.paged_decode_plan.argtypes = [P, c.c_int32, c.c_int32, c.c_int32, c.c_int32,
                                    c.POINTER(c.c_int32), c.POINTER(c.c_int32), c.POINTER(c.c_size_t)]
    L.paged_decode_attention.restype = c.c_int
    L.paged_decode_attention.argtypes = [P, c.c_int, P, c.c_int32, P, c.c_int32, P, c.c_int32,
                                         c.c_int32, c.c_int32, c.c_float, c.c_int32, c.c_int, P,
                                         c.c_size_t, P, P]
    L.paged_multi_query_plan.restype = c.c_int
    L.paged_multi_query_plan.argtypes = [P, c.c_int32, c.c_int32, c.c_int32, c.c_int32, c.c_int32,
                                         c.POINTER(c.c_int32), c.POINTER(c.c_int32), c.POINTER(c.c_size_t)]
    L.paged_multi_query_attention.restype = c.c_int
    L.paged_multi_query_attention.argtypes = [P, c.c_int, P, c.c_int32, P, c.c_int32, P, c.c_int32, c.c_int32,
                                              c.c_int32, c.c_int32, c.c_float, c.c_int32, c.c_int, P,
                                              c.c_size_t, P, P]
    L.paged_multi_query_algo.restype = c.c_int32
    L.paged_multi_query_algo.argtypes = [P, c.c_int32, c.c_int32, c.c_int32, c.c_int]
    L.paged_decode_append_attention.restype = c.c_int
    L.paged_decode_append_attention.argtypes = [P, c.c_int, P, P, c.c_int, P, c.c_int32, P, c.c_int32, P,
                                                c.c_int32, c.c_int32, c.c_int32, c.c_float, c.c_int32, c.c_int,
                                                P, c.c_size_t, P, P]
    L.paged_decode_attention_static_ws.restype = c.c_int
    L.paged_decode_attention_static_ws.argtypes = [P, c.c_int, P, c.c_int32, P, c.c_int32, P, c.c_int32,
                                                   c.c_int32, c.c_int32, c.c_float, c.c_int32, c.c_int, P, P]
    L.paged_decode_algo.restype = c.c_int32
    L.paged_decode_algo.argtypes = [P, c.c_int32, c.c_int]
    L.pkv_set_first_wait_limit_for_testing.restype = None
    L.pkv_set_first_wait_limit_for_testing.argtypes = [c.c_int32, c.c_int32]
    L.pkv_status_string.restype = c.c_char_p
    L.pkv_status_string.argtypes = [c.c_int]
    L.pkv_last_cuda_error.restype = c.c_char_p
    L.pkv_last_cuda_error.argtypes = []
    _lib = L
    return L


def _check(rc: int, what: str):
    if rc != 0:
        raise PkvError(rc, what)


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return PKV_F32
    if t == torch.bfloat16:
        return PKV_BF16
    if t in (torch.float8_e4m3fn, torch.uint8):
        return PKV_FP8_E4M3
    raise ValueError("unsupported dtype %s" % t)


_POOL_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16, "fp8": torch.uint8}
_POOL_CODE = {"f32": PKV_F32, "bf16": PKV_BF16, "fp8": PKV_FP8_E4M3}


def _stream_ptr(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t: torch.Tensor, name: str, dtype=None) -> ctypes.c_void_p:
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return ctypes.c_void_p(t.data_ptr())


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, kv_dtype: str) -> int:
    return int(lib().kv_bytes_per_token(num_layers, num_kv_heads, head_dim, _POOL_CODE[kv_dtype]))


class KVPool:
    """K and V pools [layers][blocks][kv_heads][block_size][head_dim] plus the
    library's handle.  FP8 pools hold raw E4M3 bytes (torch.uint8)."""

    def __init__(self, num_layers: int, num_blocks: int, block_size: int, num_kv_heads: int,
                 head_dim: int, kv_dtype: str, k_scale: float = 1.0, v_scale: float = 1.0,
                 device: str = "cuda", fill: Optional[int] = None):
        self.num_layers, self.num_blocks, self.block_size = num_layers, num_blocks, block_size
        self.num_kv_heads, self.head_dim, self.kv_dtype = num_kv_heads, head_dim, kv_dtype
        self.k_scale, self.v_scale = float(k_scale), float(v_scale)
        shape = (num_layers, num_blocks, num_kv_heads, block_size, head_dim)
        dt = _POOL_TORCH[kv_dtype]
        self.k = torch.empty(shape, dtype=dt, device=device)
        self.v = torch.empty(shape, dtype=dt, device=device)
        if fill is not None:
            self.k.view(torch.uint8).fill_(fill)
            self.v.view(torch.uint8).fill_(fill)
        self.error_word = torch.zeros(1, dtype=torch.int32, device=device)
        self._desc = PoolDesc(num_layers, num_blocks, block_size, num_kv_heads, head_dim,
                              _POOL_CODE[kv_dtype], self.k_scale, self.v_scale, self.k.data_ptr(),
                              self.v.data_ptr(), self.error_word.data_ptr())
        h = ctypes.c_void_p()
        _check(lib().kv_pool_create(ctypes.byref(self._desc), ctypes.byref(h)), "kv_pool_create")
        self.handle = h

    @property
    def tensor_bytes(self) -> int:
        return int(lib().kv_pool_tensor_bytes(ctypes.byref(self._desc)))

    def errors(self) -> int:
        """Read (synchronously) the error bits the kernels have set."""
        return int(self.error_word.item())

    def clear_errors(self):
        self.error_word.zero_()

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            lib().kv_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def kv_append(pool: KVPool, layer: int, k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
              stream=None) -> None:
    """Write k, v [T, Hkv, D] (f32 or bf16) into the pool at slot_mapping [T] (int64)."""
    T = slot_mapping.shape[0]
    if k.shape != (T, pool.num_kv_heads, pool.head_dim) or v.shape != k.shape:
        raise ValueError("k/v must be [T, num_kv_heads, head_dim]")
    if k.dtype != v.dtype:
        raise ValueError("k and v must share a dtype")
    rc = lib().kv_append(pool.handle, layer, _dev(k, "k"), _dev(v, "v"), _dtype_code(k.dtype),
                         _dev(slot_mapping, "slot_mapping", torch.int64), T, _stream_ptr(stream))
    _check(rc, "kv_append")


def decode_plan(pool: KVPool, num_seqs: int, num_q_heads: int, max_seq_len: int,
                split_tokens: int = 0) -> Tuple[int, int, int]:
    """(split_tokens used, number of splits, workspace bytes)."""
    S, NS, ws = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_size_t()
    _check(lib().paged_decode_plan(pool.handle, num_seqs, num_q_heads, max_seq_len, split_tokens,
                                   ctypes.byref(S), ctypes.byref(NS), ctypes.byref(ws)),
           "paged_decode_plan")
    return S.value, NS.value, ws.value


def decode_algo(pool: KVPool, num_q_heads: int, algo: str = "auto") -> str:
    """Name of the kernel design a call with this request would run."""
    r = lib().paged_decode_algo(pool.handle, num_q_heads // pool.num_kv_heads, ALGOS[algo])
    if r < 0:
        raise PkvError(2, "paged_decode_algo")
    return ALGO_NAMES[r]


def workspace_for(pool: KVPool, num_seqs: int, num_q_heads: int, max_seq_len: int,
                  split_tokens: int = 0) -> Optional[torch.Tensor]:
    _, _, ws = decode_plan(pool, num_seqs, num_q_heads, max_seq_len, split_tokens)
    if ws == 0:
        return None
    # the leading per-sequence counters must start at zero
    return torch.zeros(ws, dtype=torch.uint8, device=pool.k.device)


def paged_decode_attention(q: torch.Tensor, pool: KVPool, layer: int, block_tables: torch.Tensor,
                           seq_lens: torch.Tensor, max_seq_len: int, scale: float,
                           out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                           split_tokens: int = 0, algo: str = "auto", stream=None) -> torch.Tensor:
    """out[b, hq] = softmax(scale * q[b, hq] . K^T) V over the first seq_lens[b]
    tokens of sequence b, gathered through block_tables [B, max_blocks] (int32)."""
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = workspace_for(pool, B, Hq, max_seq_len, split_tokens)
    ws_ptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None else ctypes.c_void_p()
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib().paged_decode_attention(
        _dev(q, "q"), _dtype_code(q.dtype), pool.handle, layer, _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(seq_lens, "seq_lens", torch.int32), B, Hq, max_seq_len, float(scale),
        split_tokens, ALGOS[algo], ws_ptr, ws_bytes, _dev(out, "out", q.dtype), _stream_ptr(stream))
    _check(rc, "paged_decode_attention")
    return out


def paged_decode_append_attention(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, pool: KVPool,
                                  layer: int, block_tables: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                                  scale: float, out: Optional[torch.Tensor] = None,
                                  workspace: Optional[torch.Tensor] = None, split_tokens: int = 0,
                                  algo: str = "auto", stream=None) -> torch.Tensor:
    """One launch: write k_new / v_new [B, Hkv, D] (bf16 or f32) at position
    seq_lens[b] - 1 of each sequence, then paged_decode_attention over
    seq_lens[b] tokens (tensor-core design only)."""
    B, Hq, D = q.shape
    if tuple(k_new.shape) != (B, pool.num_kv_heads, D) or k_new.shape != v_new.shape or k_new.dtype != v_new.dtype:
        raise ValueError("k_new / v_new must both be [num_seqs, num_kv_heads, head_dim] of one dtype")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = workspace_for(pool, B, Hq, max_seq_len, split_tokens)
    ws_ptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None else ctypes.c_void_p()
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib().paged_decode_append_attention(
        _dev(q, "q"), _dtype_code(q.dtype), _dev(k_new, "k_new"), _dev(v_new, "v_new"), _dtype_code(k_new.dtype),
        pool.handle, layer, _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _dev(seq_lens, "seq_lens", torch.int32), B, Hq, max_seq_len, float(scale), split_tokens, ALGOS[algo],
        ws_ptr, ws_bytes, _dev(out, "out", q.dtype), _stream_ptr(stream))
    _check(rc, "paged_decode_append_attention")
    return out


def paged_decode_attention_static_ws(q: torch.Tensor, pool: KVPool, layer: int, block_tables: torch.Tensor,
                                     seq_lens: torch.Tensor, max_seq_len: int, scale: float,
                                     out: Optional[torch.Tensor] = None, split_tokens: int = 0,
                                     algo: str = "auto", stream=None) -> torch.Tensor:
    """paged_decode_attention whose split partials live in the library's own
    fixed device array (no workspace argument; the call allocates nothing on
    the device beyond `out` when `out` is not given).  Calls that overlap on
    the GPU share that array and race."""
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    rc = lib().paged_decode_attention_static_ws(
        _dev(q, "q"), _dtype_code(q.dtype), pool.handle, layer, _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(seq_lens, "seq_lens", torch.int32), B, Hq, max_seq_len, float(scale),
        split_tokens, ALGOS[algo], _dev(out, "out", q.dtype), _stream_ptr(stream))
    _check(rc, "paged_decode_attention_static_ws")
    return out


def set_first_wait_limit_for_testing(polls: int, cta: int = -1) -> None:
    """Make the tensor-core decode design's first stage wait give up after
    `polls` polls in CTA `cta` (every CTA when negative) for later calls from
    this thread; polls < 0 restores the normal bound (test hook)."""
    lib().pkv_set_first_wait_limit_for_testing(int(polls), int(cta))


def multi_query_plan(pool: KVPool, num_seqs: int, num_queries: int, num_q_heads: int, max_seq_len: int,
                     split_tokens: int = 0) -> Tuple[int, int, int]:
    S, NS, ws = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_size_t()
    _check(lib().paged_multi_query_plan(pool.handle, num_seqs, num_queries, num_q_heads, max_seq_len, split_tokens,
                                        ctypes.byref(S), ctypes.byref(NS), ctypes.byref(ws)),
           "paged_multi_query_plan")
    return S.value, NS.value, ws.value


def multi_query_algo(pool: KVPool, num_queries: int, num_q_heads: int, split_tokens: int = 0,
                     algo: str = "auto") -> str:
    """Name of the kernel design a multi-query call with this request would run."""
    r = lib().paged_multi_query_algo(pool.handle, num_queries, num_q_heads, split_tokens, ALGOS[algo])
    if r < 0:
        raise PkvError(2, "no kernel design serves this request")
    return ALGO_NAMES[r]


def paged_multi_query_attention(q: torch.Tensor, pool: KVPool, layer: int, block_tables: torch.Tensor,
                                seq_lens: torch.Tensor, max_seq_len: int, scale: float,
                                out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                                split_tokens: int = 0, algo: str = "auto", stream=None) -> torch.Tensor:
    """q [B, C, Hq, D]: the last C tokens of each sequence, each attending
    causally (query c at position seq_lens[b] - C + c).  Returns [B, C, Hq, D]."""
    B, C, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        _, _, ws = multi_query_plan(pool, B, C, Hq, max_seq_len, split_tokens)
        workspace = torch.zeros(ws, dtype=torch.uint8, device=q.device) if ws else None
    ws_ptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None else ctypes.c_void_p()
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib().paged_multi_query_attention(
        _dev(q, "q"), _dtype_code(q.dtype), pool.handle, layer, _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(seq_lens, "seq_lens", torch.int32), B, C, Hq, max_seq_len, float(scale),
        split_tokens, ALGOS[algo], ws_ptr, ws_bytes, _dev(out, "out", q.dtype), _stream_ptr(stream))
    _check(rc, "paged_multi_query_attention")
    return out
