"""ctypes binding of libpe (argument marshalling only).

Every step of the layer runs in libpe's CUDA kernels; this module only passes
pointers and sizes across the C ABI declared in include/pe.h.  PyTorch is used
for device memory (the arena and the activations) and streams.  There is no
fallback: if libpe.so is missing or fails to load, every entry point raises.
"""

from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, byref, c_double, c_float, c_int32, c_size_t, c_uint32, c_uint64, c_void_p

import numpy as np

from .synth import MoEShape

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpe.so")

PE_OK, PE_ERR_INVALID, PE_ERR_UNSUPPORTED_DTYPE, PE_ERR_HOST_ALLOC, PE_ERR_CUDA, PE_ERR_RANGE, PE_ERR_ARENA = range(7)
PE_BF16, PE_FP8_BLOCK128, PE_INT4_GPTQ, PE_MXFP4, PE_NVFP4 = 0, 1, 2, 3, 4
_DTYPE = {"bf16": PE_BF16, "fp8": PE_FP8_BLOCK128, "int4": PE_INT4_GPTQ, "mxfp4": PE_MXFP4, "nvfp4": PE_NVFP4}
PE_DEVERR_NAN_LOGIT, PE_DEVERR_NOT_LOADED, PE_DEVERR_PLAN = 1, 2, 4

EXPORTS = [
    "pe_required_device_bytes", "pe_slots_for_budget", "pe_get_row_layout", "pe_max_waves", "pe_create",
    "pe_create_external",
    "pe_create_shared",
    "pe_load_host_expert", "pe_host_row", "pe_forward", "pe_stats", "pe_read_plan", "pe_read_residency",
    "pe_read_slot", "pe_reset_residency", "pe_probe_host_link", "pe_profile_enable", "pe_profile_read",
    "pe_destroy", "pe_last_error", "pe_expert_mlp_noalloc", "pe_selftest_bounded_waits",
]


class PEConfig(ctypes.Structure):
    _fields_ = [(n, c_int32) for n in ("num_layers", "num_experts", "top_k", "num_slots", "hidden",
                                       "intermediate", "dtype", "max_tokens", "device")]


class PERowLayout(ctypes.Structure):
    _fields_ = [(n, c_uint64) for n in ("w13_offset", "w13_bytes", "s13_offset", "s13_bytes", "w2_offset",
                                        "w2_bytes", "s2_offset", "s2_bytes", "payload_bytes", "row_stride")]


class PEStats(ctypes.Structure):
    _fields_ = [(n, c_uint64) for n in ("steps", "waves", "entries", "distinct", "hits", "page_ins",
                                        "cold_fills", "bytes_paged")] + [("error_word", c_uint32),
                                                                          ("reserved", c_uint32)]


class PEPlanView(ctypes.Structure):
    _fields_ = [("plan_expert", POINTER(c_int32)), ("plan_slot", POINTER(c_int32)),
                ("plan_count", POINTER(c_int32)), ("topk_id", POINTER(c_int32)), ("topk_w", POINTER(c_float)),
                ("entry_slot", POINTER(c_int32)), ("entry_wave", POINTER(c_int32)), ("num_waves", c_int32)]


PROF_KINDS = 12


class PEProfile(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p * PROF_KINDS), ("launches", c_uint64 * PROF_KINDS),
                ("total_ms", c_double * PROF_KINDS)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libpe.so (built in-tree by ``host_paged_expert_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libpe.so is not built ({LIB_PATH}); run host_paged_expert_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    cfgp = POINTER(PEConfig)
    L.pe_required_device_bytes.argtypes = [cfgp]
    L.pe_required_device_bytes.restype = c_size_t
    L.pe_slots_for_budget.argtypes = [cfgp, c_size_t]
    L.pe_slots_for_budget.restype = c_int32
    L.pe_get_row_layout.argtypes = [cfgp, POINTER(PERowLayout)]
    L.pe_max_waves.argtypes = [cfgp, c_int32]
    L.pe_max_waves.restype = c_int32
    L.pe_create.argtypes = [cfgp, c_void_p, c_size_t, POINTER(c_void_p)]
    L.pe_create_shared.argtypes = [cfgp, c_void_p, c_size_t, c_void_p, POINTER(c_void_p)]
    L.pe_create_external.argtypes = [cfgp, c_void_p, c_size_t, c_void_p, c_size_t, c_int32, POINTER(c_void_p)]
    L.pe_load_host_expert.argtypes = [c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p]
    L.pe_host_row.argtypes = [c_void_p, c_int32, c_int32]
    L.pe_host_row.restype = c_void_p
    L.pe_forward.argtypes = [c_void_p, c_int32, c_void_p, c_void_p, c_void_p, c_int32, c_void_p]
    L.pe_stats.argtypes = [c_void_p, c_int32, POINTER(PEStats)]
    L.pe_read_plan.argtypes = [c_void_p, c_int32, c_int32, POINTER(PEPlanView)]
    L.pe_read_residency.argtypes = [c_void_p, c_int32, c_void_p, c_void_p, c_void_p, c_void_p]
    L.pe_read_slot.argtypes = [c_void_p, c_int32, c_int32, c_void_p, c_size_t]
    L.pe_reset_residency.argtypes = [c_void_p, c_void_p]
    L.pe_probe_host_link.argtypes = [c_void_p, c_void_p, c_size_t, c_int32, c_void_p, POINTER(c_double),
                                     POINTER(c_double)]
    L.pe_profile_enable.argtypes = [c_void_p, c_int32]
    L.pe_profile_read.argtypes = [c_void_p, POINTER(PEProfile)]
    L.pe_destroy.argtypes = [c_void_p]
    L.pe_destroy.restype = None
    L.pe_expert_mlp_noalloc.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32,
                                         c_void_p]
    L.pe_last_error.argtypes = [c_void_p]
    L.pe_last_error.restype = ctypes.c_char_p
    for name in EXPORTS:
        getattr(L, name)  # every declared entry point must be exported
    _lib = L
    return L


class PEError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"libpe status {status}: {msg}")
        self.status = status


def make_config(shape: MoEShape, max_tokens: int, device: int = 0) -> PEConfig:
    return PEConfig(shape.num_layers, shape.num_experts, shape.top_k, shape.num_slots, shape.hidden,
                    shape.intermediate, _DTYPE[shape.dtype], max_tokens,
                    device)


def required_device_bytes(shape: MoEShape, max_tokens: int) -> int:
    cfg = make_config(shape, max_tokens)
    return int(lib().pe_required_device_bytes(byref(cfg)))


def selftest_bounded_waits(poll_limit: int = 1 << 16) -> list[int]:
    """Error words of the three bounded-wait kinds run on never-true
    conditions (each must read PE_DEVERR_TIMEOUT)."""
    out = (ctypes.c_uint32 * 3)()
    st = lib().pe_selftest_bounded_waits(ctypes.c_uint32(poll_limit), out)
    if st != PE_OK:
        raise PEError(st, lib().pe_last_error(None).decode())
    return [int(v) for v in out]


def slots_for_budget(shape: MoEShape, max_tokens: int, budget_bytes: int) -> int:
    """Largest K whose whole arena fits the device-memory budget (0: none)."""
    cfg = make_config(shape, max_tokens)
    return int(lib().pe_slots_for_budget(byref(cfg), c_size_t(budget_bytes)))


def host_store_bytes(shape: MoEShape) -> int:
    """Bytes of a host store for this shape: L * E * row_stride."""
    return shape.num_layers * shape.num_experts * row_layout(shape)["row_stride"]


def row_layout(shape: MoEShape) -> dict:
    cfg = make_config(shape, 1)
    r = PERowLayout()
    st = lib().pe_get_row_layout(byref(cfg), byref(r))
    if st != PE_OK:
        raise PEError(st, "invalid config")
    return {n: int(getattr(r, n)) for n, _ in PERowLayout._fields_}


def max_waves(shape: MoEShape, num_tokens: int) -> int:
    cfg = make_config(shape, max(1, num_tokens))
    return int(lib().pe_max_waves(byref(cfg), num_tokens))


def _ptr(t) -> int:
    return t.data_ptr()


def _stream_ptr(stream) -> int | None:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class PagedMoE:
    """A stack of paged MoE layers on one GPU (wraps a libpe handle)."""

    def __init__(self, shape: MoEShape, max_tokens: int, device: int = 0, store_owner: "PagedMoE | None" = None,
                 host_store=None, filled: bool = False):
        """``store_owner``: read that handle's host store.  ``host_store``: an
        object with ``ptr`` and ``nbytes`` (e.g. a SharedHostStore) to use as
        the host store; ``filled`` marks every expert in it loaded."""
        import torch

        self.shape = shape
        self.max_tokens = max_tokens
        self.device = device
        self._L = lib()
        self.cfg = make_config(shape, max_tokens, device)
        n = int(self._L.pe_required_device_bytes(byref(self.cfg)))
        if n == 0:
            raise PEError(PE_ERR_INVALID, "invalid configuration")
        self.arena = torch.empty(n, dtype=torch.uint8, device=f"cuda:{device}")
        h = c_void_p()
        if host_store is not None:
            st = self._L.pe_create_external(byref(self.cfg), c_void_p(self.arena.data_ptr()), n,
                                            c_void_p(host_store.ptr), host_store.nbytes, int(filled), byref(h))
        elif store_owner is None:
            st = self._L.pe_create(byref(self.cfg), c_void_p(self.arena.data_ptr()), n, byref(h))
        else:
            st = self._L.pe_create_shared(byref(self.cfg), c_void_p(self.arena.data_ptr()), n,
                                          store_owner.handle, byref(h))
        if st != PE_OK:
            raise PEError(st, self._L.pe_last_error(None).decode())
        self.handle = h
        self._owner = store_owner if store_owner is not None else host_store
        self.layout = row_layout(shape)

    # -- lifecycle
    def close(self) -> None:
        if getattr(self, "handle", None):
            self._L.pe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, st: int) -> None:
        if st != PE_OK:
            raise PEError(st, self._L.pe_last_error(self.handle).decode())

    # -- experts
    def load_expert(self, layer: int, expert: int, row: dict) -> None:
        w13 = np.ascontiguousarray(row["w13"])
        w2 = np.ascontiguousarray(row["w2"])
        s13 = row.get("s13")
        s2 = row.get("s2")
        dt = self.shape.dtype
        if dt in ("mxfp4", "nvfp4"):
            # byte grids; NVFP4 puts the tensor's fp32 scale in a 16-byte header first
            def grid(sc, g):
                sc = np.ascontiguousarray(sc, dtype=np.uint8).reshape(-1)
                if dt == "mxfp4":
                    return sc
                hdr = np.zeros(16, np.uint8)
                hdr[:4] = np.array([g], dtype=np.float32).view(np.uint8)
                return np.concatenate([hdr, sc])

            s13 = grid(s13, row.get("g13"))
            s2 = grid(s2, row.get("g2"))
        else:
            sdt = np.float16 if dt == "int4" else np.float32
            s13 = None if s13 is None else np.ascontiguousarray(s13, dtype=sdt)
            s2 = None if s2 is None else np.ascontiguousarray(s2, dtype=sdt)
        self._check(self._L.pe_load_host_expert(
            self.handle, layer, expert, w13.ctypes.data, w2.ctypes.data,
            None if s13 is None else s13.ctypes.data, None if s2 is None else s2.ctypes.data))

    def host_row(self, layer: int, expert: int) -> np.ndarray:
        """Writable numpy view (uint8) of an expert's host-store row."""
        p = self._L.pe_host_row(self.handle, layer, expert)
        if not p:
            raise PEError(PE_ERR_RANGE, "layer or expert out of range")
        n = self.layout["row_stride"]
        return np.ctypeslib.as_array((ctypes.c_uint8 * n).from_address(p))

    # -- forward
    def forward(self, layer: int, hidden, logits, out=None, stream=None):
        import torch

        T = hidden.shape[0]
        if out is None:
            out = torch.empty_like(hidden)
        self._check(self._L.pe_forward(self.handle, layer, c_void_p(_ptr(hidden)), c_void_p(_ptr(logits)),
                                       c_void_p(_ptr(out)), T, c_void_p(_stream_ptr(stream))))
        return out

    def forward_ptr(self, layer: int, hidden_ptr: int, logits_ptr: int, out_ptr: int, num_tokens: int,
                    stream_ptr: int) -> None:
        self._check(self._L.pe_forward(self.handle, layer, c_void_p(hidden_ptr), c_void_p(logits_ptr),
                                       c_void_p(out_ptr), num_tokens, c_void_p(stream_ptr)))

    # -- inspection
    def stats(self, layer: int = -1) -> dict:
        s = PEStats()
        self._check(self._L.pe_stats(self.handle, layer, byref(s)))
        return {n: int(getattr(s, n)) for n, _ in PEStats._fields_ if n != "reserved"}

    def read_plan(self, layer: int, num_tokens: int) -> dict:
        W = max_waves(self.shape, num_tokens)
        K = self.shape.num_slots
        n = num_tokens * self.shape.top_k
        arrs = {
            "plan_expert": np.zeros((W, K), np.int32), "plan_slot": np.zeros((W, K), np.int32),
            "plan_count": np.zeros(W, np.int32), "topk_id": np.zeros((num_tokens, self.shape.top_k), np.int32),
            "topk_w": np.zeros((num_tokens, self.shape.top_k), np.float32),
            "entry_slot": np.zeros((num_tokens, self.shape.top_k), np.int32),
            "entry_wave": np.zeros((num_tokens, self.shape.top_k), np.int32),
        }
        v = PEPlanView()
        for name, a in arrs.items():
            ctype = c_float if a.dtype == np.float32 else c_int32
            setattr(v, name, a.ctypes.data_as(POINTER(ctype)))
        self._check(self._L.pe_read_plan(self.handle, layer, num_tokens, byref(v)))
        arrs["num_waves"] = int(v.num_waves)
        return arrs

    def read_residency(self, layer: int) -> dict:
        K, E = self.shape.num_slots, self.shape.num_experts
        se = np.zeros(K, np.int32)
        tk = np.zeros(K, np.uint32)
        es = np.zeros(E, np.int32)
        ck = np.zeros(1, np.uint32)
        self._check(self._L.pe_read_residency(self.handle, layer, se.ctypes.data, tk.ctypes.data,
                                              es.ctypes.data, ck.ctypes.data))
        return {"slot_expert": se, "slot_tick": tk, "expert_slot": es, "clock": int(ck[0])}

    def read_slot(self, layer: int, slot: int, nbytes: int | None = None) -> np.ndarray:
        n = self.layout["row_stride"] if nbytes is None else nbytes
        buf = np.zeros(n, np.uint8)
        self._check(self._L.pe_read_slot(self.handle, layer, slot, buf.ctypes.data, n))
        return buf

    def reset_residency(self, stream=None) -> None:
        self._check(self._L.pe_reset_residency(self.handle, c_void_p(_stream_ptr(stream))))

    def probe_host_link(self, nbytes: int, iters: int = 5, stream=None) -> tuple[float, float]:
        import torch

        dst = torch.empty(nbytes, dtype=torch.uint8, device=f"cuda:{self.device}")
        ce, kn = c_double(), c_double()
        self._check(self._L.pe_probe_host_link(self.handle, c_void_p(dst.data_ptr()), nbytes, iters,
                                               c_void_p(_stream_ptr(stream)), byref(ce), byref(kn)))
        return float(ce.value), float(kn.value)

    def profile_enable(self, on: bool = True) -> None:
        self._check(self._L.pe_profile_enable(self.handle, 1 if on else 0))

    def profile_read(self) -> dict:
        p = PEProfile()
        self._check(self._L.pe_profile_read(self.handle, byref(p)))
        out = {}
        for i in range(PROF_KINDS):
            if p.name[i]:
                out[p.name[i].decode()] = {"launches": int(p.launches[i]), "total_ms": float(p.total_ms[i])}
        return out
