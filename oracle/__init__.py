"""fp64 CPU oracle for cached-KV attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  It shares no code with the CUDA library and imports
nothing from it.

The arithmetic lives in ``gist_attn_oracle.c`` (plain C, double precision);
this module compiles it with gcc on first use and exposes it through ctypes.
``gist_mask`` holds the training-side gist mask used by the brute-force pins;
``projections`` the linear layers on either side of the attention.

Sources are cited by page title and section:
  [Gist page]  "把 item 压成 KV：gist 能不能用在相关性任务上" (liam.page, 2026-10-30)
  [KV page]    "为什么自回归推理缓存 KV，而不缓存历史 Q？" (mcfzz.com notes)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gist_attn_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs: dict[int, ctypes.CDLL] = {}


class OraDims(ctypes.Structure):
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
        ("rope_theta", ctypes.c_double),
        ("softmax_scale", ctypes.c_double),
        ("prerotated", ctypes.c_int32),
    ]


def build(force: bool = False, plant: int = 0) -> str:
    """Compile the C oracle into oracle/_build/ (no -ffast-math).

    ``plant`` > 0 builds a copy with one deliberate mistake (see ORA_PLANT in
    the C source); only the pin-sensitivity tests ask for it.
    """
    os.makedirs(_OUT_DIR, exist_ok=True)
    path = os.path.join(_OUT_DIR, "liboracle.so" if plant == 0 else f"liboracle_plant{plant}.so")
    if (not force and os.path.exists(path)
            and os.path.getmtime(path) >= os.path.getmtime(_SRC)):
        return path
    tmp = path + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", f"-DORA_PLANT={plant}",
                           "-o", tmp, _SRC, "-lm", "-lpthread"])
    os.replace(tmp, path)
    return path


def _load(plant: int = 0):
    with _lock:
        if plant not in _libs:
            lib = ctypes.CDLL(build(plant=plant))
            P = ctypes.c_void_p
            for name in ("ora_gist_attn", "ora_gist_attn_f64"):
                fn = getattr(lib, name)
                fn.restype = ctypes.c_int
                fn.argtypes = [P, P, P, P, P, P, P, P, ctypes.c_int32, P, P,
                               ctypes.POINTER(OraDims), ctypes.c_int32]
            lib.ora_gist_attn_fp8kv.restype = ctypes.c_int
            lib.ora_gist_attn_fp8kv.argtypes = [P, P, P, P, P, P, P, P, P, ctypes.c_int32, P, P,
                                                ctypes.POINTER(OraDims), ctypes.c_int32]
            lib.ora_e4m3_to_f64.restype = ctypes.c_double
            lib.ora_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.ora_gist_attn_masked.restype = ctypes.c_int
            lib.ora_gist_attn_masked.argtypes = [P, P, P, P, P, P, P, P, ctypes.c_int32, P,
                                                 ctypes.c_int32, P, P, ctypes.POINTER(OraDims),
                                                 ctypes.c_int32]
            lib.ora_kv_store.restype = ctypes.c_int
            lib.ora_kv_store.argtypes = [P, P, P, P, P, P, ctypes.POINTER(OraDims)]
            lib.ora_kv_append.restype = ctypes.c_int
            lib.ora_kv_append.argtypes = [P, P, P, P, P, P, ctypes.POINTER(OraDims)]
            lib.ora_gather.restype = ctypes.c_int
            lib.ora_gather.argtypes = [P, P, P, P, ctypes.POINTER(OraDims)]
            lib.ora_rope.restype = None
            lib.ora_rope.argtypes = [P, ctypes.c_int, ctypes.c_double, ctypes.c_double, P]
            lib.ora_bf16_to_f64.restype = ctypes.c_double
            lib.ora_bf16_to_f64.argtypes = [ctypes.c_uint16]
            for name in ("ora_kv_bytes_per_position",):
                getattr(lib, name).restype = ctypes.c_int64
                getattr(lib, name).argtypes = [ctypes.c_int64] * 4
            lib.ora_kv_bytes_per_item.restype = ctypes.c_int64
            lib.ora_kv_bytes_per_item.argtypes = [ctypes.c_int64] * 5
            lib.ora_kv_bytes_batch.restype = ctypes.c_int64
            lib.ora_kv_bytes_batch.argtypes = [ctypes.c_int64] * 6
            _libs[plant] = lib
    return _libs[plant]


def bf16_bits(x) -> np.ndarray:
    """bf16 values as a contiguous uint16 array of their bit patterns.

    Accepts a torch bf16 tensor (any device; copied to host) or a uint16 array.
    """
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("expected bf16 bit patterns as uint16")
        return np.ascontiguousarray(x)
    import torch  # plain CPU data movement only
    if x.dtype != torch.bfloat16:
        raise TypeError(f"expected a bf16 tensor, got {x.dtype}")
    return np.ascontiguousarray(x.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16))


def _i32(x):
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x, dtype=np.int32)
    return np.ascontiguousarray(x.detach().cpu().numpy(), dtype=np.int32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def make_dims(**kw) -> OraDims:
    d = OraDims()
    d.rope_theta = 1e4
    d.softmax_scale = 0.0
    d.prerotated = 0
    d.num_layers = 1
    d.layer = 0
    for k, v in kw.items():
        if k == "flags":  # the library's flag word: bit 0 = q and k_new arrive rotated
            d.prerotated = int(v) & 1
        else:
            setattr(d, k, v)
    return d


def _f64(x):
    if x is None:
        return None
    if not isinstance(x, np.ndarray):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def gist_attn(q, k_new, v_new, kv_pool, item_ids=None, block_table=None, pos_offset=None, *,
              dims: dict, pairs=None, want_weights: bool = False, num_threads: int | None = None,
              f64_inputs: bool = False, plant: int = 0, gist_start=None, gist_len: int = 0):
    """Attention output in float64, shape [n][l][Hq][d] (n = len(pairs) or P).

    Inputs are bf16 (torch tensors or uint16 bit arrays) in the library's
    layouts; see gist_attn_oracle.c.  With ``f64_inputs`` they are float64
    arrays in the same layouts instead.  With want_weights the softmax weights
    [n][l][Hq][C+l] (zeros where masked) are returned too.  With ``gist_start``
    ([P] ints) the gist mask applies: a token after keys
    [gist_start, gist_start + gist_len) no longer sees the keys before them.
    """
    lib = _load(plant)
    D = make_dims(**dims)
    conv = _f64 if f64_inputs else bf16_bits
    qb, kb, vb = conv(q), conv(k_new), conv(v_new)
    pb = conv(kv_pool) if kv_pool is not None else None
    ids, tab, pos, sel = _i32(item_ids), _i32(block_table), _i32(pos_offset), _i32(pairs)
    n = D.num_pairs if sel is None else int(sel.shape[0])
    C = D.blocks_per_pair * D.block_len
    out = np.zeros((n, D.n_new, D.num_q_heads, D.head_dim), dtype=np.float64)
    w = (np.zeros((n, D.n_new, D.num_q_heads, C + D.n_new), dtype=np.float64)
         if want_weights else None)
    if num_threads is None:
        num_threads = len(os.sched_getaffinity(0))
    if gist_start is not None:
        if f64_inputs:
            raise ValueError("the gist mask takes bf16 inputs")
        gs = _i32(gist_start)
        rc = lib.ora_gist_attn_masked(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(pb), _ptr(ids), _ptr(tab),
                                      _ptr(pos), _ptr(gs), int(gist_len), _ptr(sel), n, _ptr(out),
                                      _ptr(w), ctypes.byref(D), int(num_threads))
    else:
        fn = lib.ora_gist_attn_f64 if f64_inputs else lib.ora_gist_attn
        rc = fn(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(pb), _ptr(ids), _ptr(tab), _ptr(pos), _ptr(sel),
                n, _ptr(out), _ptr(w), ctypes.byref(D), int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle rejected the inputs (code {rc})")
    return (out, w) if want_weights else out


def u8(x) -> np.ndarray:
    """E4M3 bytes as a contiguous uint8 array (torch float8/uint8 tensor or numpy)."""
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x, dtype=np.uint8)
    import torch
    return np.ascontiguousarray(x.detach().contiguous().cpu().view(torch.uint8).numpy())


def gist_attn_fp8kv(q, k_new, v_new, kv_pool_e4m3, kv_scale, item_ids=None, block_table=None,
                    pos_offset=None, *, dims: dict, pairs=None, num_threads: int | None = None):
    """Attention with the cached segment stored as E4M3 bytes times one fp32 scale per
    (block, layer, K|V, KV head); float64 output [n][l][Hq][d]."""
    lib = _load()
    D = make_dims(**dims)
    qb, kb, vb = bf16_bits(q), bf16_bits(k_new), bf16_bits(v_new)
    pb = u8(kv_pool_e4m3) if kv_pool_e4m3 is not None else None
    sc = None
    if kv_scale is not None:
        sc = kv_scale if isinstance(kv_scale, np.ndarray) else kv_scale.detach().cpu().numpy()
        sc = np.ascontiguousarray(sc, dtype=np.float32)
    ids, tab, pos, sel = _i32(item_ids), _i32(block_table), _i32(pos_offset), _i32(pairs)
    n = D.num_pairs if sel is None else int(sel.shape[0])
    out = np.zeros((n, D.n_new, D.num_q_heads, D.head_dim), dtype=np.float64)
    if num_threads is None:
        num_threads = len(os.sched_getaffinity(0))
    rc = lib.ora_gist_attn_fp8kv(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(pb), _ptr(sc), _ptr(ids),
                                 _ptr(tab), _ptr(pos), _ptr(sel), n, _ptr(out), None,
                                 ctypes.byref(D), int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle rejected the inputs (code {rc})")
    return out


def e4m3_to_f64(byte: int) -> float:
    return float(_load().ora_e4m3_to_f64(int(byte)))


def gather(kv_pool, item_ids=None, block_table=None, *, dims: dict):
    """Bit-exact cached rows per pair: uint16 [P][Hkv][2][C][d]; also the return code."""
    lib = _load()
    D = make_dims(**dims)
    pb = bf16_bits(kv_pool)
    ids, tab = _i32(item_ids), _i32(block_table)
    C = D.blocks_per_pair * D.block_len
    dst = np.zeros((D.num_pairs, D.num_kv_heads, 2, C, D.head_dim), dtype=np.uint16)
    rc = lib.ora_gather(_ptr(pb), _ptr(ids), _ptr(tab), _ptr(dst), ctypes.byref(D))
    return dst, rc


def rope(x: np.ndarray, pos: float, theta: float = 1e4, plant: int = 0) -> np.ndarray:
    """The oracle's rotate-half RoPE of one vector (float64)."""
    lib = _load(plant)
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    lib.ora_rope(_ptr(x), int(x.shape[0]), float(pos), float(theta), _ptr(y))
    return y


def bf16_to_f64(bits: int) -> float:
    return float(_load().ora_bf16_to_f64(int(bits)))


def kv_bytes_per_position(L, Hkv, d, b) -> int:
    return int(_load().ora_kv_bytes_per_position(L, Hkv, d, b))


def kv_bytes_per_item(L, Hkv, d, k, b) -> int:
    return int(_load().ora_kv_bytes_per_item(L, Hkv, d, k, b))


def kv_bytes_batch(B, L, T, Hkv, d, b) -> int:
    return int(_load().ora_kv_bytes_batch(B, L, T, Hkv, d, b))


def block_mass(weights: np.ndarray, blocks_per_pair: int, block_len: int) -> np.ndarray:
    """Per-block attention mass of decode weights [n][1][Hq][C+1] -> [n][Hq][blocks]:
    the sum of the softmax weights over each cached block's rows (the new token's
    own key belongs to no block)."""
    C = blocks_per_pair * block_len
    w = weights[:, 0, :, :C].reshape(weights.shape[0], weights.shape[2], blocks_per_pair, block_len)
    return w.sum(axis=-1)


def kv_append(k_new, v_new, kv_pool, block_table, slot, pos_offset=None, *, dims: dict):
    """A copy of the pool (uint16 bf16 bits) with each sequence's new K (rotated,
    rounded to bf16) and V written at its slot; also the return code."""
    lib = _load()
    D = make_dims(**dims)
    pool = bf16_bits(kv_pool).copy()
    kb, vb = bf16_bits(k_new), bf16_bits(v_new)
    tab, sl, pos = _i32(block_table), _i32(slot), _i32(pos_offset)
    rc = lib.ora_kv_append(_ptr(kb), _ptr(vb), _ptr(pool), _ptr(tab), _ptr(sl), _ptr(pos),
                           ctypes.byref(D))
    return pool, rc


def kv_store(k_new, v_new, kv_pool, item_ids, first_row, store_pos=None, *, dims: dict):
    """A copy of the pool (uint16 bf16 bits) with each pair's rows
    first_row .. first_row + block_len - 1 stored as its item's cache entry at
    dims["layer"] (K rotated at store_pos + t, default t, rounded to bf16; V
    copied); also the return code."""
    lib = _load()
    D = make_dims(**dims)
    pool = bf16_bits(kv_pool).copy()
    kb, vb = bf16_bits(k_new), bf16_bits(v_new)
    ids, fr, sp = _i32(item_ids), _i32(first_row), _i32(store_pos)
    rc = lib.ora_kv_store(_ptr(kb), _ptr(vb), _ptr(pool), _ptr(ids), _ptr(fr), _ptr(sp),
                          ctypes.byref(D))
    return pool, rc
