"""Seeded synthetic inputs: random-init weights and uniform prompt ids.

This module holds no arithmetic of the decoding method.  It is the one place
both sides draw their inputs from: the CPU oracle takes the numpy arrays made
here, the CUDA path fills device buffers with the same bits through the small
``libdllm_synth`` library, which implements the same counter-based generator on
the GPU (tests check the two bit for bit).

Generator (counter-based, one 64-bit word per element):

* SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014; constants as in Vigna's public-domain
  ``splitmix64.c``): ``out(i) = mix(key + (i + 1) * 0x9E3779B97F4A7C15)`` with
  ``mix(z) = z ^ z>>30, *0xBF58476D1CE4E5B9, ^ >>27, *0x94D049BB133111EB, ^ >>31``.
* Per-tensor key: ``key = out_seed(code)`` = the ``code``-th output of the
  SplitMix64 stream seeded with the global seed, ``code = (kind << 16) | layer``.
* Approximate normal: Irwin-Hall sum of the word's four 16-bit fields,
  ``z = u0 + u1 + u2 + u3 - 131070`` (an exact integer with variance ~65536^2/3),
  then ``w = float32(z) * c`` with ``c = float32(std * sqrt(3) / 65536)``, plus an
  optional float32 ``offset`` (1.0 for RMSNorm gains when drawn randomly), then
  round-to-nearest-even to bf16.  Every step is an exact or a single correctly
  rounded IEEE operation, so the GPU reproduces the bits.
* Uniform token id in [0, V): ``((out >> 32) * V) >> 32`` (Lemire's
  multiply-shift).
"""
from __future__ import annotations

import ctypes
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .configs import ModelConfig

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK64 = (1 << 64) - 1

# tensor kinds: the "kind" field of the per-tensor stream code
KIND = {
    "embed": 1, "attn_norm": 2, "wq": 3, "wk": 4, "wv": 5, "wo": 6,
    "ffn_norm": 7, "wg": 8, "wu": 9, "wd": 10, "final_norm": 11, "lm_head": 12,
    "prompt": 13,
}
LAYER_TENSORS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "wg", "wu", "wd")
NORM_TENSORS = ("attn_norm", "ffn_norm", "final_norm")


def mix64_int(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def splitmix64_stream(seed: int, n: int) -> list[int]:
    """First n outputs of the sequential SplitMix64 generator seeded with ``seed``."""
    return [mix64_int(seed + (i + 1) * 0x9E3779B97F4A7C15) for i in range(n)]


def stream_key(seed: int, kind: str, layer: int = 0) -> int:
    code = (KIND[kind] << 16) | layer
    return mix64_int(seed + (code + 1) * 0x9E3779B97F4A7C15)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def raw_words(key: int, start: int, count: int) -> np.ndarray:
    idx = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(np.uint64(key) + idx * GAMMA)


def normal_scale(std: float) -> np.float32:
    return np.float32(std * math.sqrt(3.0) / 65536.0)


def _normal_chunk(key: int, start: int, count: int, c: np.float32, offset: np.float32) -> np.ndarray:
    u = raw_words(key, start, count)
    m16 = np.uint64(0xFFFF)
    s = (u & m16) + ((u >> np.uint64(16)) & m16) + ((u >> np.uint64(32)) & m16) + (u >> np.uint64(48))
    z = (s.astype(np.int64) - 131070).astype(np.float32)
    w = z * c
    if offset != 0:
        w = w + offset
    bits = w.view(np.uint32)
    rounded = (bits + np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


_POOL: ThreadPoolExecutor | None = None


def _pool() -> ThreadPoolExecutor:
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1))
    return _POOL


def normal_bf16(key: int, count: int, std: float, offset: float = 0.0, start: int = 0) -> np.ndarray:
    """bf16 bit patterns (uint16) of ``count`` draws, elements start..start+count-1."""
    c = normal_scale(std)
    off = np.float32(offset)
    chunk = 1 << 22
    if count <= chunk:
        return _normal_chunk(key, start, count, c, off)
    out = np.empty(count, dtype=np.uint16)

    def work(lo: int) -> None:
        hi = min(count, lo + chunk)
        out[lo:hi] = _normal_chunk(key, start + lo, hi - lo, c, off)

    list(_pool().map(work, range(0, count, chunk)))
    return out


def uniform_ids(key: int, count: int, vocab: int, start: int = 0) -> np.ndarray:
    u = raw_words(key, start, count)
    with np.errstate(over="ignore"):
        return (((u >> np.uint64(32)) * np.uint64(vocab)) >> np.uint64(32)).astype(np.int32)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------- tensors

def tensor_shape(cfg: ModelConfig, name: str) -> tuple[int, ...]:
    d, f, v = cfg.d_model, cfg.d_ffn, cfg.vocab
    return {
        "embed": (v + 1, d), "attn_norm": (d,), "wq": (d, d), "wk": (d, d), "wv": (d, d),
        "wo": (d, d), "ffn_norm": (d,), "wg": (f, d), "wu": (f, d), "wd": (d, f),
        "final_norm": (d,), "lm_head": (v, d),
    }[name]


def tensor_spec(cfg: ModelConfig, name: str, random_norms: bool) -> tuple[float, float] | None:
    """(std, offset) of a tensor's draw; None means the constant 1.0 (RMSNorm gain)."""
    if name in NORM_TENSORS:
        return (0.1, 1.0) if random_norms else None
    if name == "lm_head":
        return (cfg.lm_std, 0.0)
    return (cfg.init_std, 0.0)


def tensor_bf16(cfg: ModelConfig, seed: int, name: str, layer: int = 0,
                random_norms: bool = False, rows: slice | None = None) -> np.ndarray:
    """One logical weight tensor as bf16 bits, row-major [out][in].

    ``rows`` restricts the draw to a row range (the counter makes any slice cheap).
    """
    shape = tensor_shape(cfg, name)
    spec = tensor_spec(cfg, name, random_norms)
    row_len = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    r0, r1 = (0, shape[0]) if rows is None else (rows.start or 0, rows.stop if rows.stop is not None else shape[0])
    count = (r1 - r0) * row_len
    if spec is None:
        out = np.full(count, 0x3F80, dtype=np.uint16)  # bf16(1.0)
    else:
        std, off = spec
        out = normal_bf16(stream_key(seed, name, layer), count, std, off, start=r0 * row_len)
    return out.reshape((r1 - r0,) + tuple(shape[1:]))


def prompts(cfg: ModelConfig, seed: int, batch: int, prompt_len: int, first_seq: int = 0) -> np.ndarray:
    """Uniform prompt ids [batch][prompt_len]; sequence i draws elements i*P .. i*P+P-1."""
    key = stream_key(seed + 1, "prompt", 0)
    ids = uniform_ids(key, batch * prompt_len, cfg.vocab, start=first_seq * prompt_len)
    return ids.reshape(batch, prompt_len)


def all_tensors(cfg: ModelConfig, seed: int, random_norms: bool = False):
    """Yield (name, layer, bf16 bits) for every tensor, in the canonical file order."""
    yield "embed", 0, tensor_bf16(cfg, seed, "embed")
    for layer in range(cfg.n_layers):
        for name in LAYER_TENSORS:
            yield name, layer, tensor_bf16(cfg, seed, name, layer, random_norms)
    yield "final_norm", 0, tensor_bf16(cfg, seed, "final_norm", 0, random_norms)
    yield "lm_head", 0, tensor_bf16(cfg, seed, "lm_head")


FILE_MAGIC = b"DLLMW001"


def write_weight_file(path: str, cfg: ModelConfig, seed: int, random_norms: bool = False) -> None:
    """Write the flat weight file read by ``dllm_load``.

    Layout: 8-byte magic, int32[6] {n_layers, d_model, n_heads, head_dim, d_ffn,
    vocab}, float32[2] {rope_theta, norm_eps}, then every tensor's bf16 bits in
    the order of :func:`all_tensors` (row-major, no padding).
    """
    hdr = np.array([cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.head_dim, cfg.d_ffn, cfg.vocab], dtype=np.int32)
    flt = np.array([cfg.rope_theta, cfg.norm_eps], dtype=np.float32)
    with open(path, "wb") as fh:
        fh.write(FILE_MAGIC)
        fh.write(hdr.tobytes())
        fh.write(flt.tobytes())
        for _, _, bits in all_tensors(cfg, seed, random_norms):
            fh.write(np.ascontiguousarray(bits).tobytes())


# --------------------------------------------------------------------------- device fill

_SYNTH_LIB = None


def _synth_lib():
    global _SYNTH_LIB
    if _SYNTH_LIB is None:
        path = os.path.join(os.path.dirname(__file__), "_lib", "libdllm_synth.so")
        if not os.path.exists(path):
            raise RuntimeError(f"libdllm_synth.so is not built ({path}); run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        lib.dllm_synth_fill_normal_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                                    ctypes.c_float, ctypes.c_float, ctypes.c_int64, ctypes.c_void_p]
        lib.dllm_synth_fill_normal_bf16.restype = ctypes.c_int
        lib.dllm_synth_fill_const_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint16, ctypes.c_void_p]
        lib.dllm_synth_fill_const_bf16.restype = ctypes.c_int
        lib.dllm_synth_fill_ids.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int32,
                                            ctypes.c_int64, ctypes.c_void_p]
        lib.dllm_synth_fill_ids.restype = ctypes.c_int
        _SYNTH_LIB = lib
    return _SYNTH_LIB


def device_fill_tensor(dst_ptr: int, cfg: ModelConfig, seed: int, name: str, layer: int = 0,
                       random_norms: bool = False, stream: int = 0) -> None:
    """Fill a device buffer with the same bits as :func:`tensor_bf16` (whole tensor)."""
    lib = _synth_lib()
    count = int(np.prod(tensor_shape(cfg, name)))
    spec = tensor_spec(cfg, name, random_norms)
    if spec is None:
        rc = lib.dllm_synth_fill_const_bf16(ctypes.c_void_p(dst_ptr), count, 0x3F80, ctypes.c_void_p(stream))
    else:
        std, off = spec
        rc = lib.dllm_synth_fill_normal_bf16(ctypes.c_void_p(dst_ptr), count, stream_key(seed, name, layer),
                                             float(normal_scale(std)), float(np.float32(off)), 0,
                                             ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError(f"device fill of {name}[{layer}] failed: cuda error {rc}")


def device_fill_prompts(dst_ptr: int, cfg: ModelConfig, seed: int, batch: int, prompt_len: int,
                        first_seq: int = 0, stream: int = 0) -> None:
    lib = _synth_lib()
    rc = lib.dllm_synth_fill_ids(ctypes.c_void_p(dst_ptr), batch * prompt_len, stream_key(seed + 1, "prompt", 0),
                                 cfg.vocab, first_seq * prompt_len, ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError(f"device fill of prompts failed: cuda error {rc}")
