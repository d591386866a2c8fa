"""ctypes binding of libgistattn.so -- argument marshalling only.

Every function here checks dtypes/devices of torch tensors, passes their raw
pointers to the C ABI (include/gist_attn.h) and turns a negative return code
into GistAttnError.  All computation runs in the library's CUDA kernels; there
is no fallback: without the built library every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libgistattn.so")

OK, ERR_NULL, ERR_DIMS, ERR_UNSUPPORTED, ERR_ALIGN, ERR_LAUNCH, ERR_SCRATCH = 0, -1, -2, -3, -4, -5, -6
NOALLOC_SCRATCH_BYTES = 64 << 20  # GIST_ATTN_NOALLOC_SCRATCH_BYTES
STATUS_BAD_BLOCK, STATUS_TIMEOUT, STATUS_RANGE = 1, 2, 4
FLAG_PREROTATED = 1
FLAG_TEST_WITHHOLD = 2  # tests of the timeout path only (see the header)
# gist_attn_route: entry points and the kernels they run (GIST_ATTN_ENTRY_* / _ROUTE_*)
ENTRY_FWD, ENTRY_FWD_WS, ENTRY_FP8KV, ENTRY_BLOCK_MASS, ENTRY_GIST_MASK = 0, 1, 2, 3, 4
ROUTES = {0: "none", 1: "prefill_tc", 2: "prefill_long", 3: "prefill_stream", 4: "staged",
          5: "decode_long", 6: "decode_short", 7: "decode_gqa", 8: "decode"}

EXPORTS = ("gist_attn_fwd", "gist_attn_workspace_bytes", "gist_attn_fwd_ws", "gist_attn_fwd_noalloc", "gist_attn_fwd_fp8kv", "gist_attn_fwd_block_mass", "gist_kv_append",
           "gist_attn_fwd_gist_mask", "gist_kv_store", "gist_qkv_rope", "gist_out_proj",
           "gist_attn_gather_debug", "gist_kv_bytes_per_position", "gist_kv_bytes_per_item",
           "gist_kv_bytes_batch", "gist_attn_status_string", "gist_attn_route")


class GistAttnError(RuntimeError):
    def __init__(self, code: int, text: str):
        super().__init__(f"gist_attn error {code}: {text}")
        self.code = code


class Dims(ctypes.Structure):
    """Mirror of gist_attn_dims."""
    _fields_ = [
        ("num_pairs", ctypes.c_int32),
        ("n_new", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("block_len", ctypes.c_int32),
        ("blocks_per_pair", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("num_layers", ctypes.c_int32),
        ("layer", ctypes.c_int32),
        ("rope_theta", ctypes.c_float),
        ("softmax_scale", ctypes.c_float),
        ("status", ctypes.c_void_p),
        ("flags", ctypes.c_int32),
    ]


_lock = threading.Lock()
_lib = None


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load the built library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(
                    f"{p} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
            lib = ctypes.CDLL(p)
            V = ctypes.c_void_p
            lib.gist_attn_fwd.restype = ctypes.c_int
            lib.gist_attn_fwd.argtypes = [V, V, V, V, V, V, V, V, ctypes.POINTER(Dims), V]
            lib.gist_attn_workspace_bytes.restype = ctypes.c_size_t
            lib.gist_attn_workspace_bytes.argtypes = [ctypes.POINTER(Dims)]
            lib.gist_attn_fwd_ws.restype = ctypes.c_int
            lib.gist_attn_fwd_ws.argtypes = [V, V, V, V, V, V, V, V, V, ctypes.c_size_t,
                                             ctypes.POINTER(Dims), V]
            lib.gist_attn_fwd_noalloc.restype = ctypes.c_int
            lib.gist_attn_fwd_noalloc.argtypes = [V, V, V, V, V, V, V, V, ctypes.POINTER(Dims), V]
            lib.gist_attn_fwd_fp8kv.restype = ctypes.c_int
            lib.gist_attn_fwd_fp8kv.argtypes = [V, V, V, V, V, V, V, V, V, ctypes.POINTER(Dims), V]
            lib.gist_attn_fwd_block_mass.restype = ctypes.c_int
            lib.gist_attn_fwd_block_mass.argtypes = [V, V, V, V, V, V, V, V, ctypes.POINTER(Dims), V]
            lib.gist_kv_append.restype = ctypes.c_int
            lib.gist_kv_append.argtypes = [V, V, V, V, V, V, ctypes.POINTER(Dims), V]
            lib.gist_attn_fwd_gist_mask.restype = ctypes.c_int
            lib.gist_attn_fwd_gist_mask.argtypes = [V, V, V, V, V, V, V, V, ctypes.c_int, V,
                                                    ctypes.POINTER(Dims), V]
            lib.gist_kv_store.restype = ctypes.c_int
            lib.gist_kv_store.argtypes = [V, V, V, V, V, V, ctypes.POINTER(Dims), V]
            lib.gist_qkv_rope.restype = ctypes.c_int
            lib.gist_qkv_rope.argtypes = [V, V, V, V, V, V, ctypes.c_int, ctypes.POINTER(Dims), V]
            lib.gist_out_proj.restype = ctypes.c_int
            lib.gist_out_proj.argtypes = [V, V, V, ctypes.c_int, ctypes.POINTER(Dims), V]
            lib.gist_attn_gather_debug.restype = ctypes.c_int
            lib.gist_attn_gather_debug.argtypes = [V, V, V, V, ctypes.POINTER(Dims), V]
            lib.gist_kv_bytes_per_position.restype = ctypes.c_size_t
            lib.gist_kv_bytes_per_position.argtypes = [ctypes.c_int] * 4
            lib.gist_kv_bytes_per_item.restype = ctypes.c_size_t
            lib.gist_kv_bytes_per_item.argtypes = [ctypes.c_int] * 5
            lib.gist_kv_bytes_batch.restype = ctypes.c_size_t
            lib.gist_kv_bytes_batch.argtypes = [ctypes.c_int] * 6
            lib.gist_attn_status_string.restype = ctypes.c_char_p
            lib.gist_attn_status_string.argtypes = [ctypes.c_int]
            lib.gist_attn_route.restype = ctypes.c_int
            lib.gist_attn_route.argtypes = [ctypes.c_int, ctypes.POINTER(Dims)]
            _lib = lib
    return _lib


def status_string(code: int) -> str:
    return load_library().gist_attn_status_string(int(code)).decode()


def make_dims(d: dict, status: torch.Tensor | None = None) -> Dims:
    out = Dims()
    for name, _ in Dims._fields_:
        if name == "status":
            continue
        setattr(out, name, d.get(name, 0) if name == "flags" else d[name])
    if status is not None:
        _check(status, torch.int32, "status")
        out.status = status.data_ptr()
    return out


def _check(t, dtype, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise TypeError(f"{name} must be contiguous")


def _ptr(t, dtype, name):
    if t is None:
        return None
    _check(t, dtype, name)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _raise(rc):
    if rc != OK:
        raise GistAttnError(rc, status_string(rc))


def gist_attn_fwd(q, k_new, v_new, kv_pool, item_ids=None, block_table=None, pos_offset=None,
                  out=None, *, dims: dict, status: torch.Tensor | None = None, stream=None):
    """One layer of cached-KV attention; returns `out` (allocated if None)."""
    lib = load_library()
    if out is None:
        out = torch.empty_like(q)
    bf, i32 = torch.bfloat16, torch.int32
    D = make_dims(dims, status)
    rc = lib.gist_attn_fwd(_ptr(q, bf, "q"), _ptr(k_new, bf, "k_new"), _ptr(v_new, bf, "v_new"),
                           _ptr(kv_pool, bf, "kv_pool"), _ptr(item_ids, i32, "item_ids"),
                           _ptr(block_table, i32, "block_table"),
                           _ptr(pos_offset, i32, "pos_offset"), _ptr(out, bf, "out"),
                           ctypes.byref(D), _stream(stream))
    _raise(rc)
    return out


def route(dims: dict, entry: int = ENTRY_FWD) -> str:
    """The kernel an entry point runs for these dimensions (a name from ROUTES),
    asked of the library on the host; raises GistAttnError where the entry
    point would refuse the shape."""
    D = make_dims(dims)
    rc = int(load_library().gist_attn_route(int(entry), ctypes.byref(D)))
    if rc < 0:
        _raise(rc)
    return ROUTES[rc]


def workspace_bytes(dims: dict) -> int:
    """Device bytes gist_attn_fwd_ws wants for these dimensions (0: none)."""
    D = make_dims(dims)
    return int(load_library().gist_attn_workspace_bytes(ctypes.byref(D)))


def gist_attn_fwd_ws(q, k_new, v_new, kv_pool, item_ids=None, block_table=None, pos_offset=None,
                     out=None, workspace=None, *, dims: dict, status: torch.Tensor | None = None,
                     stream=None):
    """gist_attn_fwd with a caller-owned device workspace (a uint8 tensor of at
    least workspace_bytes(dims) bytes, or None); returns `out`."""
    lib = load_library()
    if out is None:
        out = torch.empty_like(q)
    bf, i32 = torch.bfloat16, torch.int32
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _check(workspace, torch.uint8, "workspace")
        ws_ptr, ws_bytes = ctypes.c_void_p(workspace.data_ptr()), workspace.numel()
    D = make_dims(dims, status)
    rc = lib.gist_attn_fwd_ws(_ptr(q, bf, "q"), _ptr(k_new, bf, "k_new"), _ptr(v_new, bf, "v_new"),
                              _ptr(kv_pool, bf, "kv_pool"), _ptr(item_ids, i32, "item_ids"),
                              _ptr(block_table, i32, "block_table"),
                              _ptr(pos_offset, i32, "pos_offset"), _ptr(out, bf, "out"), ws_ptr,
                              ws_bytes, ctypes.byref(D), _stream(stream))
    _raise(rc)
    return out


def gist_attn_fwd_noalloc(q, k_new, v_new, kv_pool, item_ids=None, block_table=None,
                          pos_offset=None, out=None, *, dims: dict,
                          status: torch.Tensor | None = None, stream=None):
    """gist_attn_fwd_ws for callers that cannot allocate: the scratch is the
    library's fixed device array (NOALLOC_SCRATCH_BYTES), so no workspace is
    passed.  `out` must be given by such a caller (None allocates it here, for
    convenience only).  Returns `out`."""
    lib = load_library()
    if out is None:
        out = torch.empty_like(q)
    bf, i32 = torch.bfloat16, torch.int32
    D = make_dims(dims, status)
    rc = lib.gist_attn_fwd_noalloc(_ptr(q, bf, "q"), _ptr(k_new, bf, "k_new"),
                                   _ptr(v_new, bf, "v_new"), _ptr(kv_pool, bf, "kv_pool"),
                                   _ptr(item_ids, i32, "item_ids"),
                                   _ptr(block_table, i32, "block_table"),
                                   _ptr(pos_offset, i32, "pos_offset"), _ptr(out, bf, "out"),
                                   ctypes.byref(D), _stream(stream))
    _raise(rc)
    return out


def gist_attn_fwd_fp8kv(q, k_new, v_new, kv_pool_e4m3, kv_scale, item_ids=None, block_table=None,
                        pos_offset=None, out=None, *, dims: dict, status: torch.Tensor | None = None,
                        stream=None):
    """gist_attn_fwd with an E4M3 pool (torch.float8_e4m3fn or uint8) and fp32 scales
    [num_blocks][L][2][Hkv]; returns `out` (allocated if None)."""
    lib = load_library()
    if out is None:
        out = torch.empty_like(q)
    bf, i32 = torch.bfloat16, torch.int32
    if kv_pool_e4m3 is not None and kv_pool_e4m3.dtype not in (torch.float8_e4m3fn, torch.uint8):
        raise TypeError("kv_pool_e4m3 must be float8_e4m3fn or uint8")
    pool_ptr = None
    if kv_pool_e4m3 is not None:
        _check(kv_pool_e4m3, kv_pool_e4m3.dtype, "kv_pool_e4m3")
        pool_ptr = ctypes.c_void_p(kv_pool_e4m3.data_ptr())
    D = make_dims(dims, status)
    rc = lib.gist_attn_fwd_fp8kv(_ptr(q, bf, "q"), _ptr(k_new, bf, "k_new"), _ptr(v_new, bf, "v_new"),
                                 pool_ptr, _ptr(kv_scale, torch.float32, "kv_scale"),
                                 _ptr(item_ids, i32, "item_ids"), _ptr(block_table, i32, "block_table"),
                                 _ptr(pos_offset, i32, "pos_offset"), _ptr(out, bf, "out"),
                                 ctypes.byref(D), _stream(stream))
    _raise(rc)
    return out


def gist_attn_fwd_block_mass(q, k_new, v_new, kv_pool, block_table, pos_offset=None, out=None,
                             block_mass=None, *, dims: dict, status=None, stream=None):
    """Decode step plus per-block attention mass [P][Hq][blocks_per_pair]; returns (out, mass)."""
    lib = load_library()
    if out is None:
        out = torch.empty_like(q)
    if block_mass is None:
        block_mass = torch.empty((dims["num_pairs"], dims["num_q_heads"], dims["blocks_per_pair"]),
                                 dtype=torch.float32, device=q.device)
    bf, i32 = torch.bfloat16, torch.int32
    D = make_dims(dims, status)
    rc = lib.gist_attn_fwd_block_mass(_ptr(q, bf, "q"), _ptr(k_new, bf, "k_new"), _ptr(v_new, bf, "v_new"),
                                      _ptr(kv_pool, bf, "kv_pool"), _ptr(block_table, i32, "block_table"),
                                      _ptr(pos_offset, i32, "pos_offset"), _ptr(out, bf, "out"),
                                      _ptr(block_mass, torch.float32, "block_mass"), ctypes.byref(D),
                                      _stream(stream))
    _raise(rc)
    return out, block_mass


def gist_kv_append(k_new, v_new, kv_pool, block_table, slot, pos_offset=None, *, dims: dict,
                   status=None, stream=None):
    """Writes the new token's rotated K and its V into kv_pool (in place)."""
    lib = load_library()
    bf, i32 = torch.bfloat16, torch.int32
    D = make_dims(dims, status)
    rc = lib.gist_kv_append(_ptr(k_new, bf, "k_new"), _ptr(v_new, bf, "v_new"), _ptr(kv_pool, bf, "kv_pool"),
                            _ptr(block_table, i32, "block_table"), _ptr(slot, i32, "slot"),
                            _ptr(pos_offset, i32, "pos_offset"), ctypes.byref(D), _stream(stream))
    _raise(rc)
    return kv_pool


def gist_attn_fwd_gist_mask(q, k_new, v_new, kv_pool=None, item_ids=None, block_table=None,
                            pos_offset=None, gist_start=None, gist_len: int = 0, out=None, *,
                            dims: dict, status=None, stream=None):
    """gist_attn_fwd under the gist mask (gist_start int32 [P] required); returns `out`."""
    lib = load_library()
    if out is None:
        out = torch.empty_like(q)
    bf, i32 = torch.bfloat16, torch.int32
    D = make_dims(dims, status)
    rc = lib.gist_attn_fwd_gist_mask(_ptr(q, bf, "q"), _ptr(k_new, bf, "k_new"), _ptr(v_new, bf, "v_new"),
                                     _ptr(kv_pool, bf, "kv_pool"), _ptr(item_ids, i32, "item_ids"),
                                     _ptr(block_table, i32, "block_table"),
                                     _ptr(pos_offset, i32, "pos_offset"),
                                     _ptr(gist_start, i32, "gist_start"), int(gist_len),
                                     _ptr(out, bf, "out"), ctypes.byref(D), _stream(stream))
    _raise(rc)
    return out


def gist_kv_store(k_new, v_new, kv_pool, item_ids, first_row, store_pos=None, *, dims: dict,
                  status=None, stream=None):
    """Writes each pair's k gist rows (K rotated, V copied) into kv_pool (in place)."""
    lib = load_library()
    bf, i32 = torch.bfloat16, torch.int32
    D = make_dims(dims, status)
    rc = lib.gist_kv_store(_ptr(k_new, bf, "k_new"), _ptr(v_new, bf, "v_new"), _ptr(kv_pool, bf, "kv_pool"),
                           _ptr(item_ids, i32, "item_ids"), _ptr(first_row, i32, "first_row"),
                           _ptr(store_pos, i32, "store_pos"), ctypes.byref(D), _stream(stream))
    _raise(rc)
    return kv_pool


def gist_qkv_rope(x, w_qkv, pos_offset=None, q=None, k_new=None, v_new=None, *, dims: dict,
                  status=None, stream=None):
    """QKV projection of x [P][l][d_model] with q and k rotated in the epilogue;
    returns (q, k_new, v_new) for gist_attn_fwd with flags=FLAG_PREROTATED."""
    lib = load_library()
    P, l, Hq, Hkv, d = (dims["num_pairs"], dims["n_new"], dims["num_q_heads"], dims["num_kv_heads"],
                        dims["head_dim"])
    dev = x.device
    if q is None:
        q = torch.empty((P, l, Hq, d), dtype=torch.bfloat16, device=dev)
    if k_new is None:
        k_new = torch.empty((P, l, Hkv, d), dtype=torch.bfloat16, device=dev)
    if v_new is None:
        v_new = torch.empty((P, l, Hkv, d), dtype=torch.bfloat16, device=dev)
    bf, i32 = torch.bfloat16, torch.int32
    D = make_dims(dims, status)
    rc = lib.gist_qkv_rope(_ptr(x, bf, "x"), _ptr(w_qkv, bf, "w_qkv"), _ptr(pos_offset, i32, "pos_offset"),
                           _ptr(q, bf, "q"), _ptr(k_new, bf, "k_new"), _ptr(v_new, bf, "v_new"),
                           int(x.shape[-1]), ctypes.byref(D), _stream(stream))
    _raise(rc)
    return q, k_new, v_new


def gist_out_proj(attn_out, w_o, y=None, *, dims: dict, status=None, stream=None):
    """y [P][l][d_model] = attn_out [P][l][Hq][d] . w_o^T (w_o [d_model][Hq d])."""
    lib = load_library()
    d_model = int(w_o.shape[0])
    if y is None:
        y = torch.empty((dims["num_pairs"], dims["n_new"], d_model), dtype=torch.bfloat16,
                        device=attn_out.device)
    D = make_dims(dims, status)
    rc = lib.gist_out_proj(_ptr(attn_out, torch.bfloat16, "attn_out"), _ptr(w_o, torch.bfloat16, "w_o"),
                           _ptr(y, torch.bfloat16, "y"), d_model, ctypes.byref(D), _stream(stream))
    _raise(rc)
    return y


def gist_attn_gather_debug(kv_pool, item_ids=None, block_table=None, dst=None, *, dims: dict,
                           status: torch.Tensor | None = None, stream=None):
    """Cached rows per pair, bit for bit: bf16 [P][Hkv][2][C][d]."""
    lib = load_library()
    C = dims["block_len"] * dims["blocks_per_pair"]
    if dst is None:
        dst = torch.empty((dims["num_pairs"], dims["num_kv_heads"], 2, C, dims["head_dim"]),
                          dtype=torch.bfloat16, device=kv_pool.device)
    D = make_dims(dims, status)
    rc = lib.gist_attn_gather_debug(_ptr(kv_pool, torch.bfloat16, "kv_pool"),
                                    _ptr(item_ids, torch.int32, "item_ids"),
                                    _ptr(block_table, torch.int32, "block_table"),
                                    _ptr(dst, torch.bfloat16, "dst"), ctypes.byref(D),
                                    _stream(stream))
    _raise(rc)
    return dst


def kv_bytes_per_position(L, Hkv, d, elem_bytes) -> int:
    return int(load_library().gist_kv_bytes_per_position(L, Hkv, d, elem_bytes))


def kv_bytes_per_item(L, Hkv, d, k, elem_bytes) -> int:
    return int(load_library().gist_kv_bytes_per_item(L, Hkv, d, k, elem_bytes))


def kv_bytes_batch(B, L, T, Hkv, d, elem_bytes) -> int:
    return int(load_library().gist_kv_bytes_batch(B, L, T, Hkv, d, elem_bytes))
