"""ctypes binding of libdllm.so (include/dllm.h): argument marshalling only.

Every step of the decoding path runs in the library's CUDA kernels; this
module converts numpy arrays / device pointers and raises ``DllmError`` on a
non-OK status.  It raises at first use if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import synth
from .configs import ModelConfig

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libdllm.so")

OK, EINVAL, ENOMEM, ECUDA, EIO, ESTATE, ETIMEOUT, ECANCELLED = range(8)
EVENT_REFRESH, EVENT_STEP, EVENT_COMMIT_FORWARD = 0, 1, 2
CACHE_NONE, CACHE_PREFIX, CACHE_DUAL = 0, 1, 2
MODES = {"none": CACHE_NONE, "prefix": CACHE_PREFIX, "dual": CACHE_DUAL}
SEL_THRESHOLD, SEL_FIXED_K, SEL_FACTOR, SEL_BUDGET, SEL_SCHEDULE = 0, 1, 2, 3, 4
PREC_SPLIT, PREC_BF16 = 0, 1
TENSOR_IDS = {"embed": 1, "attn_norm": 2, "wq": 3, "wk": 4, "wv": 5, "wo": 6, "ffn_norm": 7, "wg": 8, "wu": 9,
              "wd": 10, "final_norm": 11, "lm_head": 12}
KERNEL_CLASSES = ("embed", "qkv_gemm", "attention", "o_gemm", "gateup_gemm", "down_gemm", "lm_head_gemm",
                  "merge_select", "refresh_embed", "refresh_qkv_gemm", "refresh_attention", "refresh_o_gemm",
                  "refresh_gateup_gemm", "refresh_down_gemm", "persistent_step", "unused_15")


TIMELINE_SLOTS = 10   # per (CTA, phase) entries of dllm_read_step_timeline


class DllmError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"dllm status {status}: {msg}")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("d_model", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("d_ffn", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("rope_theta", ctypes.c_float), ("norm_eps", ctypes.c_float)]


class Select(ctypes.Structure):
    _fields_ = [("policy", ctypes.c_int32), ("tau", ctypes.c_float), ("k", ctypes.c_int32),
                ("factor", ctypes.c_float)]


class Stats(ctypes.Structure):
    _fields_ = [("wall_ms", ctypes.c_double), ("refresh_ms", ctypes.c_double), ("step_ms", ctypes.c_double),
                ("steps", ctypes.c_int32), ("refreshes", ctypes.c_int32), ("blocks", ctypes.c_int32),
                ("max_steps_per_block", ctypes.c_int32), ("committed", ctypes.c_int64),
                ("tau_bar", ctypes.c_double), ("kernel_launches", ctypes.c_int64),
                ("fused_steps", ctypes.c_int32), ("reserved", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {f: getattr(self, f) for f, _ in self._fields_}


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
# int32 (*)(void* user, int32 event, int32 block_idx, int32 step_in_block)
RunHook = ctypes.CFUNCTYPE(ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32)
_I64 = ctypes.c_int64
_F = ctypes.c_float

# name -> (restype, argtypes): every entry point of include/dllm.h
SIGNATURES = {
    "dllm_model_create": (_I32, [ctypes.POINTER(Config), ctypes.POINTER(_P)]),
    "dllm_model_set_tensor": (_I32, [_P, _I32, _I32, _P, _I64, _I32]),
    "dllm_load": (_I32, [ctypes.c_char_p, ctypes.POINTER(_P)]),
    "dllm_model_config": (_I32, [_P, ctypes.POINTER(Config)]),
    "dllm_free_model": (None, [_P]),
    "dllm_state_create": (_I32, [_P, _P, _I32, _I32, _I32, _I32, _P, ctypes.POINTER(_P)]),
    "dllm_state_reset": (_I32, [_P, _P]),
    "dllm_state_set_prompts_device": (_I32, [_P, _P]),
    "dllm_free_state": (None, [_P]),
    "dllm_prefill_refresh": (_I32, [_P]),
    "dllm_denoise_step": (_I32, [_P, _I32, _F, _I32, _P]),
    "dllm_denoise_step_ex": (_I32, [_P, _I32, ctypes.POINTER(Select), _I32, _P]),
    "dllm_run": (_I32, [_P, ctypes.POINTER(Select), _I32, _I32, ctypes.POINTER(Stats)]),
    "dllm_generate": (_I32, [_P, _P, _I32, _I32, _I32, _I32, _F, _I32, _P, ctypes.POINTER(Stats)]),
    "dllm_read_state": (_I32, [_P, _P, _P, _P]),
    "dllm_read_hidden": (_I32, [_P, _P]),
    "dllm_read_kv": (_I32, [_P, _I32, _P, _P]),
    "dllm_state_set_run_hook": (_I32, [_P, RunHook, _P]),
    "dllm_state_set_trace": (_I32, [_P, _I32]),
    "dllm_read_trace": (_I32, [_P, _P, _I64, ctypes.POINTER(_I32), ctypes.POINTER(_I32)]),
    "dllm_state_set_kernel_timing": (_I32, [_P, _I32]),
    "dllm_kernel_times": (_I32, [_P, _P, _P, _P, _I32]),
    "dllm_op_gemm": (_I32, [_P, _P, _P, _P, _I32, _I32, _I32, _P]),
    "dllm_state_set_precision": (_I32, [_P, _I32]),
    "dllm_state_set_persistent": (_I32, [_P, _I32]),
    "dllm_state_set_fused_refresh": (_I32, [_P, _I32]),
    "dllm_state_set_run_ahead": (_I32, [_P, _I32]),
    "dllm_state_set_mask": (_I32, [_P, _I32]),
    "dllm_state_set_step_timeline": (_I32, [_P, _I32]),
    "dllm_read_step_timeline": (_I32, [_P, _P, _I64, ctypes.POINTER(_I32), ctypes.POINTER(_I32)]),
    "dllm_op_gemm_trace": (_I32, [_P, _P, _P, _P, _I32, _I32, _I32, _P, ctypes.POINTER(_I32), _P]),
    "dllm_op_attention": (_I32, [_P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P]),
    "dllm_staleness": (_I32, [_P, _I32, _P, _P, _P, _P]),
    "dllm_op_attention_noalloc": (_I32, [_P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P]),
    "dllm_op_attention_tc": (_I32, [_P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P]),
    "dllm_op_attention_tc_ex": (_I32, [_P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _P]),
    "dllm_op_check": (_I32, [ctypes.POINTER(_I32), _P]),
    "dllm_op_wait_probe": (_I32, [_P, _I32, _I32, _P]),
    "dllm_op_select_commit": (_I32, [_P, _P, _P, _I32, _I32, _I32, _I32, _I32, ctypes.POINTER(Select), _P, _P]),
    "dllm_last_error": (ctypes.c_char_p, []),
    "dllm_status_string": (ctypes.c_char_p, [_I32]),
    "dllm_version": (_I32, []),
}

_LIB = None


def lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run __graft_entry__.build() (needs nvcc)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def check(status: int) -> None:
    if status != OK:
        msg = lib().dllm_last_error().decode(errors="replace")
        raise DllmError(status, msg)


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def make_select(policy: int = SEL_THRESHOLD, tau: float = 0.9, k: int = 1, factor: float = 1.0) -> Select:
    return Select(policy, tau, k, factor)


def config_of(cfg: ModelConfig) -> Config:
    return Config(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.head_dim, cfg.d_ffn, cfg.vocab,
                  cfg.rope_theta, cfg.norm_eps)


class Model:
    def __init__(self, handle, cfg: ModelConfig | None = None):
        self.h = handle
        self.cfg = cfg

    @classmethod
    def create(cls, cfg: ModelConfig) -> "Model":
        h = ctypes.c_void_p()
        check(lib().dllm_model_create(ctypes.byref(config_of(cfg)), ctypes.byref(h)))
        return cls(h, cfg)

    @classmethod
    def load(cls, path: str, cfg: ModelConfig | None = None) -> "Model":
        h = ctypes.c_void_p()
        check(lib().dllm_load(path.encode(), ctypes.byref(h)))
        return cls(h, cfg)

    def set_tensor(self, name: str, layer: int, bits_or_ptr, count: int | None = None, on_device: bool = False):
        if on_device:
            check(lib().dllm_model_set_tensor(self.h, TENSOR_IDS[name], layer, ctypes.c_void_p(bits_or_ptr),
                                              count, 1))
        else:
            a = np.ascontiguousarray(bits_or_ptr, dtype=np.uint16)
            check(lib().dllm_model_set_tensor(self.h, TENSOR_IDS[name], layer, _ptr(a), a.size, 0))

    @classmethod
    def from_synth(cls, cfg: ModelConfig, seed: int = 0, random_norms: bool = False) -> "Model":
        """Random-init weights drawn on the GPU by libdllm_synth (same bits as
        the numpy generator), staged in one device buffer per tensor."""
        import torch

        m = cls.create(cfg)
        largest = max(int(np.prod(synth.tensor_shape(cfg, n))) for n in ("embed", "lm_head", "wg", "wd", "wq"))
        stage = torch.empty(largest, dtype=torch.int16, device="cuda")
        names = [("embed", 0)] + [(n, l) for l in range(cfg.n_layers) for n in synth.LAYER_TENSORS] + \
                [("final_norm", 0), ("lm_head", 0)]
        stream = torch.cuda.current_stream().cuda_stream
        for name, layer in names:
            count = int(np.prod(synth.tensor_shape(cfg, name)))
            synth.device_fill_tensor(stage.data_ptr(), cfg, seed, name, layer, random_norms, stream)
            torch.cuda.current_stream().synchronize()
            m.set_tensor(name, layer, stage.data_ptr(), count, on_device=True)
        del stage
        return m

    def free(self):
        if self.h:
            lib().dllm_free_model(self.h)
            self.h = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


class State:
    def __init__(self, model: Model, prompts: np.ndarray | None, b: int, P: int, gen_len: int, block: int,
                 stream: int | None = None):
        self.model = model
        self.b, self.P, self.gen, self.B = b, P, gen_len, block
        self.T = P + gen_len
        c = Config()
        check(lib().dllm_model_config(model.h, ctypes.byref(c)))
        self.d = c.d_model
        self.vocab = c.vocab
        self.n_layers = c.n_layers
        self.n_heads = c.n_heads
        self.head_dim = c.head_dim
        h = ctypes.c_void_p()
        pr = None if prompts is None else np.ascontiguousarray(prompts, dtype=np.int32)
        check(lib().dllm_state_create(model.h, _ptr(pr), b, P, gen_len, block,
                                      ctypes.c_void_p(stream) if stream else None, ctypes.byref(h)))
        self.h = h

    def reset(self, prompts: np.ndarray | None = None):
        pr = None if prompts is None else np.ascontiguousarray(prompts, dtype=np.int32)
        check(lib().dllm_state_reset(self.h, _ptr(pr)))

    def set_prompts_device(self, ptr: int):
        check(lib().dllm_state_set_prompts_device(self.h, ctypes.c_void_p(ptr)))

    def refresh(self):
        check(lib().dllm_prefill_refresh(self.h))

    def step(self, block_idx: int, tau: float = 0.9, mode: str | int = "dual") -> np.ndarray:
        cnt = np.zeros(self.b, dtype=np.int32)
        r = lib().dllm_denoise_step(self.h, block_idx, tau, MODES.get(mode, mode), _ptr(cnt))
        if r < 0:
            check(-r)
        return cnt

    def step_ex(self, block_idx: int, sel: Select, mode: str | int = "dual") -> np.ndarray:
        cnt = np.zeros(self.b, dtype=np.int32)
        check(lib().dllm_denoise_step_ex(self.h, block_idx, ctypes.byref(sel), MODES.get(mode, mode), _ptr(cnt)))
        return cnt

    def run(self, sel: Select | None = None, mode: str | int = "dual", refresh_interval: int = 0) -> dict:
        sel = sel or make_select()
        st = Stats()
        check(lib().dllm_run(self.h, ctypes.byref(sel), MODES.get(mode, mode), refresh_interval, ctypes.byref(st)))
        return st.as_dict()

    def set_run_hook(self, fn=None):
        """Install fn(event, block_idx, step_in_block) -> int as dllm_run's
        observer (None removes it).  A nonzero return stops the run."""
        if fn is None:
            self._hook = None
            check(lib().dllm_state_set_run_hook(self.h, RunHook(), None))
            return
        self._hook = RunHook(lambda _u, ev, j, spb: int(fn(ev, j, spb)))
        check(lib().dllm_state_set_run_hook(self.h, self._hook, None))

    def tokens(self) -> np.ndarray:
        t = np.zeros((self.b, self.T), dtype=np.int32)
        check(lib().dllm_read_state(self.h, _ptr(t), None, None))
        return t

    def read(self):
        t = np.zeros((self.b, self.T), dtype=np.int32)
        c = np.zeros((self.b, self.B), dtype=np.float32)
        a = np.zeros((self.b, self.B), dtype=np.int32)
        check(lib().dllm_read_state(self.h, _ptr(t), _ptr(c), _ptr(a)))
        return t, c, a

    def hidden(self) -> np.ndarray:
        h = np.zeros((self.b, self.B, self.d), dtype=np.float32)
        check(lib().dllm_read_hidden(self.h, _ptr(h)))
        return h

    def kv(self, layer: int):
        k = np.zeros((self.b, self.n_heads, self.T, self.head_dim), dtype=np.float32)
        v = np.zeros_like(k)
        check(lib().dllm_read_kv(self.h, layer, _ptr(k), _ptr(v)))
        return k, v

    def set_precision(self, mode: str):
        check(lib().dllm_state_set_precision(self.h, {"split": PREC_SPLIT, "bf16": PREC_BF16}[mode]))

    def set_persistent(self, on: bool):
        check(lib().dllm_state_set_persistent(self.h, 1 if on else 0))

    def set_fused_refresh(self, on: bool):
        check(lib().dllm_state_set_fused_refresh(self.h, 1 if on else 0))

    def set_run_ahead(self, on: bool):
        check(lib().dllm_state_set_run_ahead(self.h, 1 if on else 0))

    def set_mask(self, mask: str):
        check(lib().dllm_state_set_mask(self.h, {"full": 0, "block_causal": 1}[mask]))

    def set_step_timeline(self, on: bool):
        check(lib().dllm_state_set_step_timeline(self.h, 1 if on else 0))

    def step_timeline(self) -> np.ndarray:
        c = ctypes.c_int32()
        ph = ctypes.c_int32()
        check(lib().dllm_read_step_timeline(self.h, None, 0, ctypes.byref(c), ctypes.byref(ph)))
        out = np.zeros((c.value, ph.value, TIMELINE_SLOTS), dtype=np.uint64)
        check(lib().dllm_read_step_timeline(self.h, _ptr(out), out.size, ctypes.byref(c), ctypes.byref(ph)))
        return out

    def set_trace(self, on: bool):
        check(lib().dllm_state_set_trace(self.h, 1 if on else 0))

    def trace(self):
        R = ctypes.c_int32()
        p0 = ctypes.c_int32()
        check(lib().dllm_read_trace(self.h, None, 0, ctypes.byref(R), ctypes.byref(p0)))
        out = np.zeros((self.n_layers + 1, self.b * R.value, self.d), dtype=np.float32)
        check(lib().dllm_read_trace(self.h, _ptr(out), out.size, ctypes.byref(R), ctypes.byref(p0)))
        return out.reshape(self.n_layers + 1, self.b, R.value, self.d), R.value, p0.value

    def set_kernel_timing(self, on: bool):
        check(lib().dllm_state_set_kernel_timing(self.h, 1 if on else 0))

    def kernel_times(self) -> dict:
        n = len(KERNEL_CLASSES)
        ms = np.zeros(n)
        cnt = np.zeros(n, dtype=np.int64)
        by = np.zeros(n)
        check(lib().dllm_kernel_times(self.h, _ptr(ms), _ptr(cnt), _ptr(by), n))
        return {k: {"ms": float(ms[i]), "launches": int(cnt[i]), "bytes": float(by[i])}
                for i, k in enumerate(KERNEL_CLASSES)}

    def staleness(self, block_idx: int) -> dict:
        L = self.n_layers
        k = np.zeros(L, dtype=np.float32)
        v = np.zeros(L, dtype=np.float32)
        agree = ctypes.c_float()
        dconf = ctypes.c_float()
        check(lib().dllm_staleness(self.h, block_idx, _ptr(k), _ptr(v), ctypes.byref(agree), ctypes.byref(dconf)))
        return {"k_cos": k, "v_cos": v, "agree": agree.value, "max_dconf": dconf.value}

    def free(self):
        if self.h:
            lib().dllm_free_state(self.h)
            self.h = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def generate(model: Model, prompts: np.ndarray, gen_len: int, block: int, tau: float = 0.9,
             mode: str | int = "dual"):
    pr = np.ascontiguousarray(prompts, dtype=np.int32)
    b, P = pr.shape
    out = np.zeros((b, gen_len), dtype=np.int32)
    st = Stats()
    check(lib().dllm_generate(model.h, _ptr(pr), b, P, gen_len, block, tau, MODES.get(mode, mode), _ptr(out),
                              ctypes.byref(st)))
    return out, st.as_dict()


def op_gemm(W_ptr: int, X_ptr: int, Y_ptr: int, M: int, N: int, K: int, stream: int = 0, X_lo_ptr: int = 0):
    check(lib().dllm_op_gemm(ctypes.c_void_p(W_ptr), ctypes.c_void_p(X_ptr),
                             ctypes.c_void_p(X_lo_ptr) if X_lo_ptr else None, ctypes.c_void_p(Y_ptr), M, N, K,
                             ctypes.c_void_p(stream)))


def op_gemm_trace(W_ptr: int, X_ptr: int, Y_ptr: int, M: int, N: int, K: int, trace_ptr: int, stream: int = 0,
                  X_lo_ptr: int = 0) -> int:
    grid = ctypes.c_int32()
    check(lib().dllm_op_gemm_trace(ctypes.c_void_p(W_ptr), ctypes.c_void_p(X_ptr),
                                   ctypes.c_void_p(X_lo_ptr) if X_lo_ptr else None, ctypes.c_void_p(Y_ptr), M, N, K,
                                   ctypes.c_void_p(trace_ptr), ctypes.byref(grid), ctypes.c_void_p(stream)))
    return grid.value


def op_attention(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, b: int, H: int, hd: int, R: int, T: int,
                 stream: int = 0):
    check(lib().dllm_op_attention(ctypes.c_void_p(q_ptr), ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr),
                                  ctypes.c_void_p(o_ptr), b, H, hd, R, T, ctypes.c_void_p(stream)))


def op_attention_tc(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, b: int, H: int, hd: int, R: int, T: int,
                    stream: int = 0, splits: int | None = None):
    if splits is None:
        check(lib().dllm_op_attention_tc(ctypes.c_void_p(q_ptr), ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr),
                                         ctypes.c_void_p(o_ptr), b, H, hd, R, T, ctypes.c_void_p(stream)))
    else:
        check(lib().dllm_op_attention_tc_ex(ctypes.c_void_p(q_ptr), ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr),
                                            ctypes.c_void_p(o_ptr), b, H, hd, R, T, splits,
                                            ctypes.c_void_p(stream)))


def op_attention_noalloc(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, b: int, H: int, hd: int, R: int,
                         T: int, stream: int = 0):
    check(lib().dllm_op_attention_noalloc(ctypes.c_void_p(q_ptr), ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr),
                                          ctypes.c_void_p(o_ptr), b, H, hd, R, T, ctypes.c_void_p(stream)))


def op_check(stream: int = 0) -> int:
    """Raise DllmError(ETIMEOUT) if a dllm_op_* kernel gave up a bounded wait
    since the last check; returns the site code (0)."""
    site = ctypes.c_int32()
    check(lib().dllm_op_check(ctypes.byref(site), ctypes.c_void_p(stream)))
    return site.value


def op_wait_probe(flag_ptr: int, need: int, limit_us: int, stream: int = 0) -> int:
    """Status of the bounded-wait probe (OK or ETIMEOUT), without raising."""
    return int(lib().dllm_op_wait_probe(ctypes.c_void_p(flag_ptr), need, limit_us, ctypes.c_void_p(stream)))


def op_select_commit(conf_ptr: int, arg_ptr: int, x_ptr: int, b: int, T: int, blk_start: int, B: int,
                     mask_id: int, sel: Select, count_ptr: int, stream: int = 0):
    check(lib().dllm_op_select_commit(ctypes.c_void_p(conf_ptr), ctypes.c_void_p(arg_ptr), ctypes.c_void_p(x_ptr),
                                      b, T, blk_start, B, mask_id, ctypes.byref(sel), ctypes.c_void_p(count_ptr),
                                      ctypes.c_void_p(stream)))
