"""ctypes binding of libcac.so (include/cac.h): argument marshalling only.

Every computation happens in the CUDA library; this module converts Python
objects to pointers and sizes, allocates output tensors with torch (device
memory is plumbing, not compute) and turns status codes into exceptions.  If
the library is not built it raises instead of falling back to anything.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int, c_int32, c_longlong, c_size_t, c_void_p

import numpy as np

from .config import ModelConfig, DTYPE_BF16, MEL_TAIL

# CAC_LIB=checked selects the CAC_CHECKED build (libcac_checked.so, built with
# build.build(checked=True)); the default build otherwise.
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                        "libcac_checked.so" if os.environ.get("CAC_LIB") == "checked" else "libcac.so")

CAC_OK = 0
ERRORS = {-1: "CAC_E_INVAL", -2: "CAC_E_ALIGN", -3: "CAC_E_STATE", -4: "CAC_E_NOMEM", -5: "CAC_E_CUDA",
          -6: "CAC_E_DEVICE", -7: "CAC_E_NONFINITE", -8: "CAC_E_TIMEOUT", -9: "CAC_E_UNSUPPORTED",
          -10: "CAC_E_LIMIT"}

# every symbol include/cac.h declares
SYMBOLS = ["cac_weights_size", "cac_model_create", "cac_model_create_palette", "cac_model_destroy", "cac_pool_create", "cac_pool_destroy",
           "cac_stream_create", "cac_stream_destroy", "cac_stream_reset", "cac_stream_push", "cac_stream_push_host",
           "cac_stream_push_host_async",
           "cac_stream_flush", "cac_stream_flush_frames", "cac_encode_offline", "cac_stream_get_state",
           "cac_stream_set_state", "cac_pool_check", "cac_model_check", "cac_pool_set_graphs",
           "cac_pool_launch_count", "cac_pool_set_chains", "cac_pool_sub_batches", "cac_pool_check_guards",
           "cac_build_checked", "cac_op_bounds_selftest", "cac_pool_set_trace", "cac_pool_read_trace", "cac_pool_set_profile",
           "cac_pool_read_profile", "cac_profile_classes", "cac_profile_class_name", "cac_strerror",
           "cac_op_gemm_bf16", "cac_encode_offline_noalloc",
           # include/cac_decode.h
           "cac_decoder_create", "cac_decoder_destroy", "cac_decoder_reset", "cac_decoder_step",
           "cac_decoder_check", "cac_decoder_get_state",
           "cac_op_wait_selftest", "cac_op_gemm_palette",
           # include/cac_frontend.h
           "cac_frontend_create", "cac_frontend_destroy", "cac_frontend_reset", "cac_frontend_push",
           "cac_frontend_flush", "cac_frontend_get_state", "cac_frontend_schedule", "cac_frontend_tables",
           # include/cac_beam.h
           "cac_beam_create", "cac_beam_destroy", "cac_beam_reset", "cac_beam_step", "cac_beam_check",
           "cac_beam_get"]


class CacError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {ERRORS.get(code, code)} ({_lib().cac_strerror(code).decode()})")


class CacConfig(ctypes.Structure):
    _fields_ = [(n, c_int32) for n in (
        "n_layers", "d_model", "n_heads", "ff_dim", "dw_kernel", "att_left", "att_chunk", "mel_bins",
        "joint_dim", "dtype", "right_context", "emit_frames", "lookahead_frames", "gemm_simt")]


class CacDecConfig(ctypes.Structure):
    _fields_ = [(n, c_int32) for n in ("vocab", "pred_dim", "joint_dim", "max_symbols")]


class CacStreamState(ctypes.Structure):
    _fields_ = [("subT", c_int32), ("Lc", c_int32), ("finished", c_int32), ("x0_rows", c_int32),
                ("mel_tail", POINTER(c_float)), ("k_cache", POINTER(c_float)), ("v_cache", POINTER(c_float)),
                ("conv_cache", POINTER(c_float)), ("x0", POINTER(c_float))]


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vp, ip, fp = c_void_p, POINTER(c_int), POINTER(c_float)
        sig = {
            "cac_weights_size": (c_size_t, [POINTER(CacConfig)]),
            "cac_model_create": (c_int, [POINTER(CacConfig), fp, c_size_t, POINTER(vp)]),
            "cac_model_create_palette": (c_int, [POINTER(CacConfig), fp, c_size_t, fp, c_size_t, POINTER(vp)]),
            "cac_model_destroy": (None, [vp]),
            "cac_pool_create": (c_int, [vp, c_int, c_int, POINTER(vp)]),
            "cac_pool_destroy": (None, [vp]),
            "cac_stream_create": (c_int, [vp, ip]),
            "cac_stream_destroy": (c_int, [vp, c_int]),
            "cac_stream_reset": (c_int, [vp, c_int, ip, vp]),
            "cac_stream_push": (c_int, [vp, c_int, ip, vp, c_int, vp, vp, ip, vp]),
            "cac_stream_push_host": (c_int, [vp, c_int, ip, vp, c_int, vp, vp, ip, vp]),
            "cac_stream_push_host_async": (c_int, [vp, c_int, ip, vp, c_int, vp, vp, ip, vp]),
            "cac_stream_flush": (c_int, [vp, c_int, ip, vp, c_int, ip, vp, vp, c_int, ip, vp]),
            "cac_stream_flush_frames": (c_int, [vp, c_int, c_int, ip]),
            "cac_encode_offline": (c_int, [vp, c_int, vp, ip, c_int, vp, vp, ip, vp]),
            "cac_encode_offline_noalloc": (c_int, [vp, c_int, vp, ip, c_int, vp, vp, ip, vp]),
            "cac_stream_get_state": (c_int, [vp, c_int, POINTER(CacStreamState)]),
            "cac_stream_set_state": (c_int, [vp, c_int, POINTER(CacStreamState)]),
            "cac_pool_check": (c_int, [vp]),
            "cac_model_check": (c_int, [vp]),
            "cac_pool_set_graphs": (c_int, [vp, c_int]),
            "cac_pool_launch_count": (c_longlong, [vp]),
            "cac_pool_set_chains": (c_int, [vp, c_int]),
            "cac_pool_sub_batches": (c_int, [vp, c_int, c_int]),
            "cac_pool_check_guards": (c_int, [vp]),
            "cac_build_checked": (c_int, []),
            "cac_op_bounds_selftest": (c_int, [vp]),
            "cac_pool_set_trace": (c_int, [vp, c_int]),
            "cac_pool_read_trace": (c_int, [vp, c_int, c_int, fp, c_size_t]),
            "cac_pool_set_profile": (c_int, [vp, c_int]),
            "cac_pool_read_profile": (c_int, [vp, c_int, POINTER(ctypes.c_double), POINTER(c_longlong)]),
            "cac_profile_classes": (c_int, []),
            "cac_profile_class_name": (c_char_p, [c_int]),
            "cac_strerror": (c_char_p, [c_int]),
            "cac_op_gemm_bf16": (c_int, [c_int, c_int, c_int, vp, vp, vp, vp, c_int, c_int, vp]),
            "cac_decoder_create": (c_int, [POINTER(CacDecConfig), fp, c_size_t, c_int, POINTER(vp)]),
            "cac_decoder_destroy": (None, [vp]),
            "cac_decoder_reset": (c_int, [vp, c_int, ip, vp]),
            "cac_decoder_step": (c_int, [vp, c_int, ip, vp, c_longlong, c_int, vp, vp, vp, vp]),
            "cac_decoder_check": (c_int, [vp]),
            "cac_decoder_get_state": (c_int, [vp, c_int, fp, fp, fp, ip]),
            "cac_op_wait_selftest": (c_int, [c_int, vp]),
            "cac_op_gemm_palette": (c_int, [c_int, c_int, c_int, vp, vp, vp, vp, vp, vp, vp]),
            "cac_frontend_create": (c_int, [c_int, POINTER(vp)]),
            "cac_frontend_destroy": (None, [vp]),
            "cac_frontend_reset": (c_int, [vp, c_int, ip]),
            "cac_frontend_push": (c_int, [vp, c_int, ip, vp, c_longlong, c_int, vp, c_longlong, c_int, ip, vp]),
            "cac_frontend_flush": (c_int, [vp, c_int, ip, vp, c_longlong, ip, vp, c_longlong, c_int, ip, vp]),
            "cac_frontend_get_state": (c_int, [vp, c_int, POINTER(c_longlong), POINTER(c_longlong), ip]),
            "cac_frontend_schedule": (c_longlong, [c_longlong, c_longlong, c_longlong, c_int]),
            "cac_frontend_tables": (c_int, [fp, fp, ip, fp]),
            "cac_beam_create": (c_int, [POINTER(CacDecConfig), fp, c_size_t, c_int, c_int, c_int, POINTER(vp)]),
            "cac_beam_destroy": (None, [vp]),
            "cac_beam_reset": (c_int, [vp, c_int, ip]),
            "cac_beam_step": (c_int, [vp, c_int, ip, vp, c_longlong, c_int, c_int, vp]),
            "cac_beam_check": (c_int, [vp]),
            "cac_beam_get": (c_int, [vp, c_int, c_int, fp, ip, ip, ip]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _LIB = L
    return _LIB


def lib():
    return _lib()


def _check(code: int, what: str):
    if code != CAC_OK:
        raise CacError(code, what)


def make_config(cfg: ModelConfig, gemm_simt: bool = False) -> CacConfig:
    return CacConfig(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.ff_dim, cfg.dw_kernel, cfg.att_left,
                     cfg.att_chunk, cfg.mel_bins, cfg.joint_dim, 1 if cfg.dtype == DTYPE_BF16 else 0,
                     cfg.right_context, cfg.emit_frames, cfg.lookahead_frames, 1 if gemm_simt else 0)


def weights_size(cfg: ModelConfig) -> int:
    c = make_config(cfg)
    return int(_lib().cac_weights_size(ctypes.byref(c)))


_IDS_CACHE: dict = {}


def _ids(ids) -> ctypes.Array:
    """ids as a C int array.  The same id list pushed again (a pool's streams,
    every step) reuses its array: the library only reads it, and building a
    256-entry ctypes array costs more than the lookup."""
    key = tuple(ids)
    arr = _IDS_CACHE.get(key)
    if arr is None:
        vals = [int(i) for i in key]
        arr = (c_int * len(vals))(*vals)
        if len(_IDS_CACHE) >= 64:
            _IDS_CACHE.clear()
        _IDS_CACHE[key] = arr
    return arr


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream=None) -> int | None:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def gemm_bf16(A, B, bias=None, splits: int = 0, out=None, stream=None, split: bool = False):
    """C = A @ B^T (+ bias) on the tcgen05 GEMM (cac_op_gemm_bf16); A [M,K], B [N,K] bf16 cuda.
    split: A is [M, 2K] = [hi | lo] and the product is (hi + lo) @ B^T."""
    import torch
    M, K = A.shape
    if split:
        K //= 2
    N = B.shape[0]
    C = out if out is not None else torch.empty(M, N, device=A.device, dtype=torch.float32)
    _check(_lib().cac_op_gemm_bf16(M, N, K, _ptr(A), _ptr(B), _ptr(bias), _ptr(C), splits, int(split),
                                   _stream(stream)), "cac_op_gemm_bf16")
    return C


class Model:
    """A model on the current CUDA device (cac_model_create)."""

    def __init__(self, cfg: ModelConfig, blob: np.ndarray, gemm_simt: bool = False, tables=None):
        """tables: optional [5 + 11 L][64] palette tables (cac_model_create_palette)."""
        self.cfg = cfg
        blob = np.ascontiguousarray(blob, dtype=np.float32)
        self._c = make_config(cfg, gemm_simt)
        h = c_void_p()
        if tables is None:
            _check(_lib().cac_model_create(ctypes.byref(self._c), blob.ctypes.data_as(POINTER(c_float)), blob.size,
                                           ctypes.byref(h)), "cac_model_create")
        else:
            t = np.ascontiguousarray(tables, dtype=np.float32)
            _check(_lib().cac_model_create_palette(ctypes.byref(self._c), blob.ctypes.data_as(POINTER(c_float)),
                                                   blob.size, t.ctypes.data_as(POINTER(c_float)), t.size,
                                                   ctypes.byref(h)), "cac_model_create_palette")
        self.h = h

    def close(self):
        if self.h:
            _lib().cac_model_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def check(self):
        _check(_lib().cac_model_check(self.h), "device status")

    def encode_offline(self, mel, mel_len, joint: bool = True, stream=None, out=None, noalloc: bool = False):
        """mel: cuda float32 [B, T_mel, 128]; returns (enc [B,T,D], joint [B,T,J] or None, out_len list).

        out: optional preallocated (enc, joint) tensors.  noalloc: use
        cac_encode_offline_noalloc (the library's fixed scratch, no device
        allocation inside the call)."""
        import torch
        B, t_mel, _ = mel.shape
        T = t_mel
        for _ in range(3):
            T = (T + 1) // 2
        if out is not None:
            enc, jt = out
        else:
            enc = torch.empty(B, T, self.cfg.d_model, device=mel.device, dtype=torch.float32)
            jt = torch.empty(B, T, self.cfg.joint_dim, device=mel.device, dtype=torch.float32) if joint else None
        out_len = (c_int * B)()
        fn = _lib().cac_encode_offline_noalloc if noalloc else _lib().cac_encode_offline
        _check(fn(self.h, B, _ptr(mel.contiguous()), _ids(mel_len), t_mel, _ptr(enc), _ptr(jt), out_len,
                  _stream(stream)), "cac_encode_offline_noalloc" if noalloc else "cac_encode_offline")
        return enc, jt, list(out_len)


class Pool:
    """Per-stream state pool (cac_pool_create) with push / flush / reset."""

    def __init__(self, model: Model, max_streams: int, max_frames_per_step: int = 8):
        self.model = model
        self.cfg = model.cfg
        h = c_void_p()
        _check(_lib().cac_pool_create(model.h, max_streams, max_frames_per_step, ctypes.byref(h)),
               "cac_pool_create")
        self.h = h

    def close(self):
        if self.h:
            _lib().cac_pool_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def create_stream(self) -> int:
        i = c_int()
        _check(_lib().cac_stream_create(self.h, ctypes.byref(i)), "cac_stream_create")
        return i.value

    def destroy_stream(self, sid: int):
        _check(_lib().cac_stream_destroy(self.h, sid), "cac_stream_destroy")

    def reset(self, ids, stream=None):
        ids = list(ids)
        if ids:
            _check(_lib().cac_stream_reset(self.h, len(ids), _ids(ids), _stream(stream)), "cac_stream_reset")

    def push_into(self, ids, mel, enc, joint, stream=None):
        """Push into caller-provided outputs; returns n_out per stream."""
        ids = list(ids)
        n_out = (c_int * len(ids))()
        _check(_lib().cac_stream_push(self.h, len(ids), _ids(ids), _ptr(mel), mel.shape[1], _ptr(enc),
                                      _ptr(joint), n_out, _stream(stream)), "cac_stream_push")
        return list(n_out)

    def push(self, ids, mel, joint: bool = True, stream=None):
        """mel: cuda float32 [n, n_mel, 128]; returns (enc [n, F, D], joint [n, F, J] or None, n_out)."""
        import torch
        n, n_mel, _ = mel.shape
        F = n_mel // 8
        enc = torch.empty(n, F, self.cfg.d_model, device=mel.device, dtype=torch.float32)
        jt = torch.empty(n, F, self.cfg.joint_dim, device=mel.device, dtype=torch.float32) if joint else None
        n_out = self.push_into(ids, mel.contiguous(), enc, jt, stream)
        return enc, jt, n_out

    def push_host(self, ids, mel, joint: bool = True, stream=None, out=None):
        """Host-buffer push (cac_stream_push_host).  mel: numpy array or CPU torch
        tensor [n, n_mel, 128] float32 (pinned tensors are copied directly);
        out: optional (enc, joint) CPU tensors / arrays to write, else new numpy
        arrays are returned."""
        ids = list(ids)
        if hasattr(mel, "data_ptr"):  # torch CPU tensor
            assert mel.dtype.is_floating_point and mel.is_contiguous() and not mel.is_cuda
            n, n_mel, _ = mel.shape
            mel_ptr = c_void_p(mel.data_ptr())
        else:
            mel = np.ascontiguousarray(mel, dtype=np.float32)
            n, n_mel, _ = mel.shape
            mel_ptr = mel.ctypes.data_as(c_void_p)
        F = n_mel // 8
        if out is not None:
            enc, jt = out
        else:
            enc = np.empty((n, F, self.cfg.d_model), dtype=np.float32)
            jt = np.empty((n, F, self.cfg.joint_dim), dtype=np.float32) if joint else None

        def addr(a):
            if a is None:
                return None
            return c_void_p(a.data_ptr()) if hasattr(a, "data_ptr") else a.ctypes.data_as(c_void_p)
        n_out = (c_int * n)()
        _check(_lib().cac_stream_push_host(self.h, n, _ids(ids), mel_ptr, n_mel, addr(enc), addr(jt), n_out,
                                           _stream(stream)), "cac_stream_push_host")
        return enc, jt, list(n_out)

    def push_host_async(self, ids, mel, out, stream=None):
        """Queued host-buffer push (cac_stream_push_host_async).  mel: pinned CPU
        torch tensor [n, n_mel, 128] float32; out: (enc, joint) pinned CPU
        tensors to receive the frames (joint may be None).  Returns n_out; the
        frames are in `out` once `stream` has passed this call's work, and
        until then mel must not change nor `out` be read."""
        ids = list(ids)
        enc, jt = out
        for t in (mel, enc, jt):
            assert t is None or (t.dtype.is_floating_point and t.is_contiguous() and not t.is_cuda)
        n, n_mel, _ = mel.shape
        n_out = (c_int * n)()
        _check(_lib().cac_stream_push_host_async(self.h, n, _ids(ids), c_void_p(mel.data_ptr()), n_mel,
                                                 c_void_p(enc.data_ptr()) if enc is not None else None,
                                                 c_void_p(jt.data_ptr()) if jt is not None else None, n_out,
                                                 _stream(stream)), "cac_stream_push_host_async")
        return list(n_out)

    def flush_frames(self, sid: int, n_mel: int) -> int:
        """Frames a flush of `n_mel` remaining mel frames emits for stream `sid`
        (held-back provisional frames included)."""
        f = c_int(0)
        _check(_lib().cac_stream_flush_frames(self.h, sid, n_mel, ctypes.byref(f)), "cac_stream_flush_frames")
        return f.value

    def flush(self, ids, mel, n_mel_each, joint: bool = True, stream=None):
        """mel: cuda float32 [n, mel_stride, 128] (or None when all n_mel_each are 0)."""
        import torch
        ids = list(ids)
        n = len(ids)
        mel_stride = 0 if mel is None else mel.shape[1]
        out_stride = max([1] + [self.flush_frames(i, m) for i, m in zip(ids, n_mel_each)])
        dev = mel.device if mel is not None else torch.device("cuda")
        enc = torch.zeros(n, out_stride, self.cfg.d_model, device=dev, dtype=torch.float32)
        jt = torch.zeros(n, out_stride, self.cfg.joint_dim, device=dev, dtype=torch.float32) if joint else None
        n_out = (c_int * n)()
        _check(_lib().cac_stream_flush(self.h, n, _ids(ids), _ptr(mel), mel_stride, _ids(n_mel_each), _ptr(enc),
                                       _ptr(jt), out_stride, n_out, _stream(stream)), "cac_stream_flush")
        return enc, jt, list(n_out)

    def get_state(self, sid: int) -> dict:
        c = self.cfg
        L, A, D = c.n_layers, c.att_left, c.d_model
        tail = np.zeros((MEL_TAIL, c.mel_bins), np.float32)
        k = np.zeros((L, A, D), np.float32)
        v = np.zeros((L, A, D), np.float32)
        conv = np.zeros((L, c.dw_kernel - 1, D), np.float32)
        fp = POINTER(c_float)
        st = CacStreamState(0, 0, 0, 0, tail.ctypes.data_as(fp), k.ctypes.data_as(fp), v.ctypes.data_as(fp),
                            conv.ctypes.data_as(fp), None)
        _check(_lib().cac_stream_get_state(self.h, sid, ctypes.byref(st)), "cac_stream_get_state")
        return {"subT": st.subT, "Lc": st.Lc, "finished": st.finished, "mel_tail": tail, "k": k, "v": v,
                "conv": conv}

    def set_state(self, sid: int, state: dict):
        fp = POINTER(c_float)
        arrs = {n: np.ascontiguousarray(state[n], dtype=np.float32) for n in ("mel_tail", "k", "v", "conv")}
        st = CacStreamState(int(state["subT"]), 0, int(state.get("finished", 0)), 0,
                            arrs["mel_tail"].ctypes.data_as(fp), arrs["k"].ctypes.data_as(fp),
                            arrs["v"].ctypes.data_as(fp), arrs["conv"].ctypes.data_as(fp), None)
        _check(_lib().cac_stream_set_state(self.h, sid, ctypes.byref(st)), "cac_stream_set_state")

    def check(self):
        _check(_lib().cac_pool_check(self.h), "device status")

    def set_graphs(self, on: bool):
        _check(_lib().cac_pool_set_graphs(self.h, 1 if on else 0), "cac_pool_set_graphs")

    def launch_count(self) -> int:
        return int(_lib().cac_pool_launch_count(self.h))

    def sub_batches(self, n_streams: int, n_frames: int) -> int:
        """Concurrent sub-batches a push of n_streams x n_frames runs as (cac_pool_sub_batches)."""
        r = int(_lib().cac_pool_sub_batches(self.h, n_streams, n_frames))
        _check(min(r, 0), "cac_pool_sub_batches")
        return r

    def check_guards(self):
        """Raise CacError(CAC_E_BOUNDS) when a kernel wrote into a pool guard zone."""
        _check(_lib().cac_pool_check_guards(self.h), "cac_pool_check_guards")

    def set_chains(self, on: bool):
        """Chained steps (default) or one launch per projection (cac_pool_set_chains)."""
        _check(_lib().cac_pool_set_chains(self.h, 1 if on else 0), "cac_pool_set_chains")

    def set_profile(self, on: bool):
        _check(_lib().cac_pool_set_profile(self.h, 1 if on else 0), "cac_pool_set_profile")

    def read_profile(self) -> dict:
        """{class name: (total ms, launches)} since the previous read (synchronizes)."""
        n = _lib().cac_profile_classes()
        ms = (ctypes.c_double * n)()
        cnt = (c_longlong * n)()
        _check(_lib().cac_pool_read_profile(self.h, n, ms, cnt), "cac_pool_read_profile")
        return {_lib().cac_profile_class_name(i).decode(): (ms[i], cnt[i]) for i in range(n)}

    def set_trace(self, on: bool):
        _check(_lib().cac_pool_set_trace(self.h, 1 if on else 0), "cac_pool_set_trace")

    def read_trace(self, layer: int, tap: int, rows: int) -> np.ndarray:
        out = np.zeros((rows, self.cfg.d_model), np.float32)
        _check(_lib().cac_pool_read_trace(self.h, layer, tap, out.ctypes.data_as(POINTER(c_float)), out.size),
               "cac_pool_read_trace")
        return out


def gemm_palette(A, packed, table, bias=None, out=None, status=None, stream=None):
    """C = A W^T (+ bias) with W[n][k] = table[6-bit index k of packed row n]
    (cac_op_gemm_palette).  A: cuda bf16 [M, K]; packed: cuda uint8 [N, 3K/4];
    table: cuda bf16 [64]; returns fp32 [M, N]."""
    import torch
    M, K = A.shape
    N = packed.shape[0]
    assert packed.shape[1] * 4 == 3 * K and A.is_contiguous() and packed.is_contiguous()
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _check(_lib().cac_op_gemm_palette(M, N, K, _ptr(A), _ptr(packed), _ptr(table), _ptr(bias), _ptr(out),
                                      _ptr(status), _stream(stream)), "cac_op_gemm_palette")
    return out


def build_checked() -> bool:
    """True when the loaded library is the CAC_CHECKED build."""
    return bool(_lib().cac_build_checked())


def bounds_selftest(stream=None) -> int:
    """Status latched by the checked build's index check on an out-of-range
    index (cac_op_bounds_selftest): CAC_E_BOUNDS (-11); CAC_E_UNSUPPORTED (-9)
    in the default build."""
    return int(_lib().cac_op_bounds_selftest(_stream(stream)))


def wait_selftest(which: int, stream=None) -> int:
    """Status latched by a bounded device wait that nothing satisfies
    (cac_op_wait_selftest): CAC_E_TIMEOUT (-8) when the wait gave up."""
    return int(_lib().cac_op_wait_selftest(int(which), _stream(stream)))


class Decoder:
    """Batched greedy RNN-T + EOU decoder on the current CUDA device
    (include/cac_decode.h): per-stream predictor state for ids 0 .. max_streams-1."""

    def __init__(self, dcfg, blob: np.ndarray, max_streams: int):
        self.cfg = dcfg
        blob = np.ascontiguousarray(blob, dtype=np.float32)
        self._c = CacDecConfig(dcfg.vocab, dcfg.pred_dim, dcfg.joint_dim, dcfg.max_symbols)
        h = c_void_p()
        _check(_lib().cac_decoder_create(ctypes.byref(self._c), blob.ctypes.data_as(POINTER(c_float)), blob.size,
                                         max_streams, ctypes.byref(h)), "cac_decoder_create")
        self.h = h
        self.max_streams = max_streams

    def close(self):
        if self.h:
            _lib().cac_decoder_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reset(self, ids, stream=None):
        _check(_lib().cac_decoder_reset(self.h, len(ids), _ids(ids), _stream(stream)), "cac_decoder_reset")

    def step_into(self, ids, z, tokens, frames, counts, stream=None):
        """z: cuda fp32 [n, T, joint_dim] (slots may be strided); outputs int32
        cuda tensors [n, T * max_symbols], [n, T * max_symbols], [n]."""
        n, T, J = z.shape
        assert J == self.cfg.joint_dim and z.stride(2) == 1 and (T <= 1 or z.stride(1) == J)
        bstride = z.stride(0) if n > 1 else T * J  # a size-1 dimension may carry any stride
        _check(_lib().cac_decoder_step(self.h, n, _ids(ids), _ptr(z), bstride, T, _ptr(tokens), _ptr(frames),
                                       _ptr(counts), _stream(stream)), "cac_decoder_step")

    def step(self, ids, z, stream=None):
        import torch
        n, T, _ = z.shape
        w = T * self.cfg.max_symbols
        tokens = torch.full((n, w), -1, dtype=torch.int32, device=z.device)
        frames = torch.full((n, w), -1, dtype=torch.int32, device=z.device)
        counts = torch.zeros(n, dtype=torch.int32, device=z.device)
        self.step_into(ids, z, tokens, frames, counts, stream)
        return tokens, frames, counts

    def check(self):
        _check(_lib().cac_decoder_check(self.h), "cac_decoder_check")

    def state(self, sid: int):
        P, J = self.cfg.pred_dim, self.cfg.joint_dim
        h, c, p = np.zeros(P, np.float32), np.zeros(P, np.float32), np.zeros(J, np.float32)
        primed = c_int(0)
        fp = POINTER(c_float)
        _check(_lib().cac_decoder_get_state(self.h, sid, h.ctypes.data_as(fp), c.ctypes.data_as(fp),
                                            p.ctypes.data_as(fp), ctypes.byref(primed)), "cac_decoder_get_state")
        return h, c, p, primed.value


def frontend_schedule(samples_before: int, frames_before: int, n_samples: int, flush: bool) -> int:
    """Frames a push (or flush) of n_samples emits (cac_frontend_schedule; host only)."""
    return int(_lib().cac_frontend_schedule(samples_before, frames_before, n_samples, 1 if flush else 0))


def frontend_tables():
    """(window [512], twiddles [256, 2], mel_start [128], mel_w [128, 16]) as the
    front-end kernel uses them (cac_frontend_tables; host only)."""
    win, tw = np.zeros(512, np.float32), np.zeros((256, 2), np.float32)
    st, mw = np.zeros(128, np.int32), np.zeros((128, 16), np.float32)
    fp, ip = POINTER(c_float), POINTER(c_int)
    _check(_lib().cac_frontend_tables(win.ctypes.data_as(fp), tw.ctypes.data_as(fp), st.ctypes.data_as(ip),
                                      mw.ctypes.data_as(fp)), "cac_frontend_tables")
    return win, tw, st, mw


class Frontend:
    """Streaming log-mel front end on the current CUDA device
    (include/cac_frontend.h): 16 kHz audio -> 128-bin log-mel frames for
    stream ids 0 .. max_streams-1."""

    N_MELS = 128

    def __init__(self, max_streams: int):
        h = c_void_p()
        _check(_lib().cac_frontend_create(max_streams, ctypes.byref(h)), "cac_frontend_create")
        self.h = h
        self.max_streams = max_streams

    def close(self):
        if self.h:
            _lib().cac_frontend_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reset(self, ids):
        _check(_lib().cac_frontend_reset(self.h, len(ids), _ids(ids)), "cac_frontend_reset")

    def _bstride(self, t, n, inner):
        if t is None:
            return 0
        assert t.stride(-1) == 1
        return t.stride(0) if n > 1 else inner  # a size-1 dimension may carry any stride

    def push_into(self, ids, audio, mel, stream=None):
        """audio: cuda fp32 [n, samples]; mel: cuda fp32 [n, max_frames, 128]
        (slots may be strided).  Returns the frames written per slot."""
        n = len(ids)
        ns = 0 if audio is None else audio.shape[1]
        max_frames = mel.shape[1]
        assert mel.shape[2] == self.N_MELS and (max_frames <= 1 or mel.stride(1) == self.N_MELS)
        out = (c_int * n)()
        _check(_lib().cac_frontend_push(self.h, n, _ids(ids), _ptr(audio), self._bstride(audio, n, ns), ns,
                                        _ptr(mel), self._bstride(mel, n, max_frames * self.N_MELS), max_frames,
                                        out, _stream(stream)), "cac_frontend_push")
        return list(out)

    def flush_into(self, ids, audio, n_samples_each, mel, stream=None):
        """Last samples (audio [n, >= max(n_samples_each)]) and every remaining frame."""
        n = len(ids)
        ns = int(max(n_samples_each)) if n else 0
        max_frames = mel.shape[1]
        assert mel.shape[2] == self.N_MELS and (max_frames <= 1 or mel.stride(1) == self.N_MELS)
        out = (c_int * n)()
        lda = 0 if audio is None else self._bstride(audio, n, audio.shape[1])
        _check(_lib().cac_frontend_flush(self.h, n, _ids(ids), _ptr(audio), lda, _ids(n_samples_each), _ptr(mel),
                                         self._bstride(mel, n, max_frames * self.N_MELS), max_frames, out,
                                         _stream(stream)), "cac_frontend_flush")
        return list(out)

    def push(self, ids, audio, max_frames=None, flush=False, n_samples_each=None, stream=None):
        """Frames of one push (or flush) as a list of cuda [frames, 128] tensors."""
        import torch
        n = len(ids)
        ns = 0 if audio is None else audio.shape[1]
        if max_frames is None:  # a push emits at most ns/160 + 1 frames, a flush up to ns/160 + 3
            ns_max = int(max(n_samples_each)) if (flush and n_samples_each is not None and n) else ns
            max_frames = ns_max // 160 + (4 if flush else 2)
        mel = torch.empty((n, max(max_frames, 1), self.N_MELS), dtype=torch.float32,
                          device=audio.device if audio is not None else "cuda")
        if flush:
            counts = self.flush_into(ids, audio, n_samples_each if n_samples_each is not None else [ns] * n, mel,
                                     stream)
        else:
            counts = self.push_into(ids, audio, mel, stream)
        return [mel[b, :counts[b]] for b in range(n)]

    def state(self, sid: int):
        """(samples received, frames emitted, finished) of one stream."""
        s, f, fin = c_longlong(0), c_longlong(0), c_int(0)
        _check(_lib().cac_frontend_get_state(self.h, sid, ctypes.byref(s), ctypes.byref(f), ctypes.byref(fin)),
               "cac_frontend_get_state")
        return s.value, f.value, fin.value


class BeamDecoder:
    """Batched MALSD RNN-T beam search on the current CUDA device
    (include/cac_beam.h) for stream ids 0 .. max_streams-1; the weights and
    config are those of the greedy decoder."""

    def __init__(self, dcfg, blob: np.ndarray, beam: int, max_streams: int, max_tokens: int = 1024):
        self.cfg, self.K, self.lmax = dcfg, beam, max_tokens
        blob = np.ascontiguousarray(blob, dtype=np.float32)
        self._c = CacDecConfig(dcfg.vocab, dcfg.pred_dim, dcfg.joint_dim, dcfg.max_symbols)
        h = c_void_p()
        _check(_lib().cac_beam_create(ctypes.byref(self._c), blob.ctypes.data_as(POINTER(c_float)), blob.size, beam,
                                      max_streams, max_tokens, ctypes.byref(h)), "cac_beam_create")
        self.h = h

    def close(self):
        if self.h:
            _lib().cac_beam_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reset(self, ids):
        _check(_lib().cac_beam_reset(self.h, len(ids), _ids(ids)), "cac_beam_reset")

    def step(self, ids, z, final: bool = False, stream=None):
        """z: cuda fp32 [n, T, joint_dim] (slots may be strided) or None with T = 0."""
        n = len(ids)
        if z is None:
            T, bstride = 0, 0
        else:
            _, T, J = z.shape
            assert J == self.cfg.joint_dim and z.stride(2) == 1 and (T <= 1 or z.stride(1) == J)
            bstride = z.stride(0) if n > 1 else T * J
        _check(_lib().cac_beam_step(self.h, n, _ids(ids), _ptr(z), bstride, T, 1 if final else 0, _stream(stream)),
               "cac_beam_step")

    def check(self):
        _check(_lib().cac_beam_check(self.h), "cac_beam_check")

    def beam(self, sid: int, score_norm: bool = True):
        """(slots as (tokens, score) or None, index of the winner)."""
        K, L = self.K, self.lmax
        sc, ln = np.zeros(K, np.float32), np.zeros(K, np.int32)
        tok = np.zeros((K, L), np.int32)
        best = c_int(-1)
        ip = POINTER(c_int)
        _check(_lib().cac_beam_get(self.h, sid, 1 if score_norm else 0, sc.ctypes.data_as(POINTER(c_float)),
                                   ln.ctypes.data_as(ip), tok.ctypes.data_as(ip), ctypes.byref(best)), "cac_beam_get")
        slots = [None if not np.isfinite(sc[k]) else (tuple(int(t) for t in tok[k, :ln[k]]), float(sc[k]))
                 for k in range(K)]
        return slots, best.value
