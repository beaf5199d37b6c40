"""B300-native quantised routed-MoE layer forward.

A thin ctypes binding of ``libmoe.so`` (see ``include/moe_layer.h``): argument
marshalling only. Every step of the layer runs in the library's CUDA kernels; there is
no CPU or PyTorch fallback. The library is loaded on first use (``lib``), and that use
fails loudly when it has not been built (``python -m quantized_moe_noaux_b300.build``).
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

__all__ = ["MoeLayer", "MoeError", "lib", "LIB_PATH", "SYMBOLS", "STAGES", "W_INT4_G32", "W_NVFP4",
           "W_BF16", "DT_F32", "DT_BF16", "PATH_AUTO", "PATH_GEMV", "PATH_GROUPED", "PATH_GENERIC"]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe.so")

W_INT4_G32, W_NVFP4, W_BF16, W_INT8_ROW, W_INT4_ROW, W_INT2_ROW = 0, 1, 2, 3, 4, 5
DT_F32, DT_BF16 = 0, 1
PATH_AUTO, PATH_GEMV, PATH_GROUPED, PATH_GENERIC = 0, 1, 2, 3

_FMT = {"int4_g32": W_INT4_G32, "nvfp4": W_NVFP4, "bf16": W_BF16, "int8_row": W_INT8_ROW,
        "int4_row": W_INT4_ROW, "int2_row": W_INT2_ROW}
_ACT = {"none": 0, "q8_0": 1}
_DT = {"f32": DT_F32, "bf16": DT_BF16}
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_OOM",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_DEVICE_CHECK"}


class MoeError(RuntimeError):
    def __init__(self, call: str, code: int):
        super().__init__(f"{call} failed: {STATUS.get(code, code)}")
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("n_group", ctypes.c_int32), ("topk_group", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32), ("routed_scaling_factor", ctypes.c_float),
                ("weight_format", ctypes.c_int32), ("shared_format", ctypes.c_int32),
                ("act_dtype", ctypes.c_int32), ("router_dtype", ctypes.c_int32),
                ("expert_top_p", ctypes.c_float), ("act_quant", ctypes.c_int32)]


class Weights(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in (
        "router_w", "bias", "gu_codes", "gu_scales", "gu_tscale", "d_codes", "d_scales",
        "d_tscale", "sh_gu", "sh_gu_scales", "sh_gu_tscale", "sh_d", "sh_d_scales", "sh_d_tscale")]


_P = ctypes.c_void_p
_I = ctypes.c_int32

# name -> (restype, argtypes): every entry point the header declares
SYMBOLS = {
    "moe_layer_create": (_I, [ctypes.POINTER(Config), ctypes.POINTER(Weights), _P,
                              ctypes.POINTER(_P)]),
    "moe_layer_forward": (_I, [_P, _P, _I, _P, _P]),
    "moe_layer_forward_host": (_I, [_P, _P, _I, _P, _P]),
    "moe_layer_get_routing": (_I, [_P, _I, _P, _P, _P, _P, _P]),
    "moe_layer_set_path": (_I, [_P, _I]),
    "moe_layer_status": (_I, [_P]),
    "moe_layer_destroy": (None, [_P]),
    "moe_layer_enable_timing": (_I, [_P, _I]),
    "moe_layer_stage_times": (_I, [_P, _P, _P]),
    "moe_layer_launch_count": (_I, [_P, _P]),
    "moe_layer_set_trace": (_I, [_P, _P, _I]),
    "moe_layer_set_wait_limit": (_I, [_P, ctypes.c_int64]),
    "moe_layer_reset_status": (_I, [_P, _P]),
    "moe_layer_set_test_activation": (_I, [_P, _I]),
    "moe_layer_set_debug_checks": (_I, [_P, _I]),
    "moe_check_routing": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "moe_test_fail_allocation": (_I, [_I]),
    "moe_layer_get_nvfp4_act": (_I, [_P, _I, _P, _P, _P, _P]),
    "moe_layer_create_cached": (_I, [ctypes.POINTER(Config), ctypes.POINTER(Weights), _I, _P,
                                     ctypes.POINTER(_P)]),
    "moe_cache_slots_for_memory": (_I, [ctypes.POINTER(Config), ctypes.c_uint64, ctypes.POINTER(_I)]),
    "moe_layer_prefetch": (_I, [_P, _P, _I, _P]),
    "moe_layer_cache_pin_hot": (_I, [_P, _I]),
    "moe_layer_cache_stats": (_I, [_P, _P]),
    "moe_layer_cache_query": (_I, [_P, _P, _P]),
    "moe_route_noalloc": (_I, [_P, _I, _I, _I, _P, _I, _P, _I, _I, _I, _I, ctypes.c_float,
                               _P, _P, _P, _P, _P]),
    "moe_status_string": (ctypes.c_char_p, [_I]),
}

# Stage slots of moe_layer_stage_times. The fused decode kernel (routing + gate/up + down +
# combine in one launch) is recorded in the third slot.
STAGES = ("routing", "act_quant", "gate_up_or_fused", "shared_gate_up", "h_quant", "down_combine", "output")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m quantized_moe_noaux_b300.build` (no fallback exists)")
    handle = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SYMBOLS.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    return handle


_lib = None


def __getattr__(name):
    if name == "lib":
        return _get_lib()
    raise AttributeError(name)


def _get_lib():
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


def _check(call: str, code: int):
    if code != 0:
        raise MoeError(call, code)


def _ptr(a) -> int | None:
    """Address of a contiguous numpy array or torch tensor (host or device)."""
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        if not a.flags.c_contiguous:
            raise ValueError("arrays must be C-contiguous")
        return a.ctypes.data
    if hasattr(a, "data_ptr"):
        if not a.is_contiguous():
            raise ValueError("tensors must be contiguous")
        return a.data_ptr()
    raise TypeError(type(a))


_torch = None


def _torch_module():
    global _torch
    if _torch is None:
        import torch
        _torch = torch
    return _torch


def _act_ptr(a, hidden: int, act_dtype: str, device: bool, name: str) -> int:
    """Address of an activation buffer, after checking that it is a contiguous [T, hidden]
    array in act_dtype (bf16: torch.bfloat16, or 16-bit integer bit patterns; f32: float32),
    in device memory for forward and prefetch and in host memory for forward_host. The
    library cannot see a buffer's size or memory kind, and a wrong one would make its
    kernels read or write outside the buffer or dereference a host address, so the binding
    refuses it before the call."""
    if isinstance(a, np.ndarray):
        if device:
            raise TypeError(f"{name}: a numpy array is host memory; pass a CUDA tensor (or use forward_host)")
        dt = a.dtype
        ok = dt == np.float32 if act_dtype == "f32" else (dt == np.uint16 or dt == np.int16)
        contiguous = a.flags.c_contiguous
    else:
        is_cuda = getattr(a, "is_cuda", None)
        if is_cuda is None:
            raise TypeError(f"{name}: {type(a)} is neither a numpy array nor a torch tensor")
        if is_cuda != device:
            raise TypeError(f"{name}: expected a {'CUDA' if device else 'host (CPU)'} tensor")
        t, dt = _torch_module(), a.dtype
        ok = dt is t.float32 if act_dtype == "f32" else (dt is t.bfloat16 or dt is t.int16)
        contiguous = a.is_contiguous()
    shape = a.shape
    if len(shape) != 2 or shape[1] != hidden:
        raise ValueError(f"{name}: expected shape [T, {hidden}], got {tuple(shape)}")
    if not ok:
        raise TypeError(f"{name}: element type {dt} does not match the layer's {act_dtype} activations")
    if not contiguous:
        raise ValueError(f"{name}: must be contiguous")
    return a.ctypes.data if isinstance(a, np.ndarray) else a.data_ptr()


def _row_bytes(fmt: str, k: int) -> tuple[int, int]:
    """(code bytes, scale bytes) of one weight row of k inputs in a storage format."""
    return {"int4_g32": (k // 2, (k // 32) * 2), "nvfp4": (k // 2, k // 16), "int8_row": (k, 4),
            "int4_row": (k // 2, 4), "int2_row": (k // 4, 4), "bf16": (2 * k, 0)}[fmt]


def weight_bytes(hidden: int, inter: int, n_experts: int, weight_format: str, shared_format: str,
                 router_dtype: str) -> dict:
    """Byte size of every weight array of a layer, as laid out in include/moe_layer.h."""
    H, I, E = hidden, inter, n_experts
    gc, gs = _row_bytes(weight_format, H)
    dc, ds = _row_bytes(weight_format, I)
    want = {"router_w": E * H * (4 if router_dtype == "f32" else 2), "bias": 4 * E,
            "gu_codes": E * 2 * I * gc, "gu_scales": E * 2 * I * gs, "d_codes": E * H * dc,
            "d_scales": E * H * ds}
    if weight_format == "nvfp4":
        want.update(gu_tscale=4 * E, d_tscale=4 * E)
    sgc, sgs = _row_bytes(shared_format, H)
    sdc, sds = _row_bytes(shared_format, I)
    if shared_format == "bf16":
        want.update(sh_gu_bf16=2 * I * sgc, sh_d_bf16=H * sdc)
    else:
        want.update(sh_gu_codes=2 * I * sgc, sh_gu_scales=2 * I * sgs, sh_d_codes=H * sdc, sh_d_scales=H * sds)
        if shared_format == "nvfp4":
            want.update(sh_gu_tscale=4, sh_d_tscale=4)
    return want


def _nbytes(a) -> int:
    return a.nbytes if isinstance(a, np.ndarray) else a.numel() * a.element_size()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


def config_from_spec(spec, max_tokens: int) -> Config:
    """The moe_config of any object with the ``synth.LayerSpec`` attribute names."""
    return Config(spec.hidden, spec.inter, spec.n_experts, spec.top_k, spec.n_group, spec.topk_group,
                  max_tokens, spec.rsf, _FMT[spec.weight_format], _FMT[spec.shared_format],
                  _DT[spec.act_dtype], _DT[spec.router_dtype], getattr(spec, "expert_top_p", 0.0),
                  _ACT[getattr(spec, "act_quant", "none")])


def cache_slots_for_memory(spec, max_tokens: int, budget_bytes: int) -> int:
    """moe_cache_slots_for_memory: the expert slots of a cached layer that fit the budget."""
    slots = ctypes.c_int32()
    cfg = config_from_spec(spec, max_tokens)
    _check("moe_cache_slots_for_memory", _get_lib().moe_cache_slots_for_memory(
        ctypes.byref(cfg), int(budget_bytes), ctypes.byref(slots)))
    return slots.value


class MoeLayer:
    """One layer: ``MoeLayer(arrays, hidden=..., ..., max_tokens=...)``.

    ``arrays`` maps the weight names of ``include/moe_layer.h`` (``router_w``, ``bias``,
    ``gu_codes``, ``gu_scales``, ``gu_tscale``, ``d_codes``, ``d_scales``, ``d_tscale``,
    and for the shared expert ``sh_gu_codes``/``sh_gu_bf16``, ``sh_gu_scales``, ...) to
    contiguous numpy arrays or torch tensors (host or device). The library copies them.
    """

    def __init__(self, arrays: dict, *, hidden: int, inter: int, n_experts: int, top_k: int,
                 n_group: int, topk_group: int, rsf: float, weight_format: str,
                 shared_format: str, act_dtype: str, router_dtype: str, max_tokens: int,
                 expert_top_p: float = 0.0, act_quant: str = "none", cache_slots: int = 0,
                 stream=None):
        self.cfg = Config(hidden, inter, n_experts, top_k, n_group, topk_group, max_tokens,
                          rsf, _FMT[weight_format], _FMT[shared_format], _DT[act_dtype],
                          _DT[router_dtype], expert_top_p, _ACT[act_quant])
        self.hidden, self.top_k, self.n_experts, self.max_tokens = hidden, top_k, n_experts, max_tokens
        self.act_dtype = act_dtype
        a = arrays
        # the library copies each array with the size its layout implies: a shorter array
        # would be read past its end (a missing one is the library's MOE_ERR_INVALID_ARG)
        for name, nb in weight_bytes(hidden, inter, n_experts, weight_format, shared_format,
                                     router_dtype).items():
            if a.get(name) is not None and _nbytes(a[name]) != nb:
                raise ValueError(f"weight array {name}: {_nbytes(a[name])} bytes, the layout needs {nb}")
        sh_gu = a.get("sh_gu_bf16") if shared_format == "bf16" else a.get("sh_gu_codes")
        sh_d = a.get("sh_d_bf16") if shared_format == "bf16" else a.get("sh_d_codes")
        w = Weights(_ptr(a["router_w"]), _ptr(a["bias"]), _ptr(a["gu_codes"]),
                    _ptr(a.get("gu_scales")), _ptr(a.get("gu_tscale")), _ptr(a["d_codes"]),
                    _ptr(a.get("d_scales")), _ptr(a.get("d_tscale")), _ptr(sh_gu),
                    _ptr(a.get("sh_gu_scales")), _ptr(a.get("sh_gu_tscale")), _ptr(sh_d),
                    _ptr(a.get("sh_d_scales")), _ptr(a.get("sh_d_tscale")))
        handle = _P()
        if cache_slots:
            # routed experts stay in host memory; HBM caches `cache_slots` of them
            _check("moe_layer_create_cached", _get_lib().moe_layer_create_cached(
                ctypes.byref(self.cfg), ctypes.byref(w), int(cache_slots), _stream(stream), ctypes.byref(handle)))
        else:
            _check("moe_layer_create", _get_lib().moe_layer_create(ctypes.byref(self.cfg), ctypes.byref(w),
                                                             _stream(stream), ctypes.byref(handle)))
        self._h = handle

    @classmethod
    def from_spec(cls, spec, arrays: dict, max_tokens: int, stream=None, cache_slots: int = 0) -> "MoeLayer":
        """Build from any object with the ``synth.LayerSpec`` attribute names."""
        return cls(arrays, hidden=spec.hidden, inter=spec.inter, n_experts=spec.n_experts,
                   top_k=spec.top_k, n_group=spec.n_group, topk_group=spec.topk_group,
                   rsf=spec.rsf, weight_format=spec.weight_format,
                   shared_format=spec.shared_format, act_dtype=spec.act_dtype,
                   router_dtype=spec.router_dtype, max_tokens=max_tokens,
                   expert_top_p=getattr(spec, "expert_top_p", 0.0),
                   act_quant=getattr(spec, "act_quant", "none"), cache_slots=cache_slots, stream=stream)

    @property
    def handle(self) -> int:
        return self._h.value

    def forward(self, x, out, stream=None):
        """out[T, H] = layer(x[T, H]) on device tensors, asynchronous on ``stream``."""
        px = _act_ptr(x, self.hidden, self.act_dtype, True, "x")
        po = _act_ptr(out, self.hidden, self.act_dtype, True, "out")
        T = x.shape[0]
        if out.shape[0] != T:
            raise ValueError(f"out has {out.shape[0]} rows for {T} tokens")
        _check("moe_layer_forward", _get_lib().moe_layer_forward(self._h, px, T, po, _stream(stream)))
        return out

    def forward_host(self, x_host, out_host, stream=None):
        """Same with host buffers (copies in, forward, copies out, synchronises)."""
        px = _act_ptr(x_host, self.hidden, self.act_dtype, False, "x_host")
        po = _act_ptr(out_host, self.hidden, self.act_dtype, False, "out_host")
        T = x_host.shape[0]
        if out_host.shape[0] != T:
            raise ValueError(f"out_host has {out_host.shape[0]} rows for {T} tokens")
        _check("moe_layer_forward_host", _get_lib().moe_layer_forward_host(self._h, px, T, po, _stream(stream)))
        return out_host

    def routing(self, T: int, stream=None) -> dict:
        """Routing of the last forward with T tokens, as host numpy arrays."""
        k, E = self.top_k, self.n_experts
        r = {"ids": np.empty((T, k), np.int32), "weights": np.empty((T, k), np.float32),
             "offsets": np.empty(E + 1, np.int32), "entries": np.empty(T * k, np.int32)}
        _check("moe_layer_get_routing", _get_lib().moe_layer_get_routing(
            self._h, T, _ptr(r["ids"]), _ptr(r["weights"]), _ptr(r["offsets"]),
            _ptr(r["entries"]), _stream(stream)))
        return r

    def set_path(self, path: int):
        _check("moe_layer_set_path", _get_lib().moe_layer_set_path(self._h, path))

    def enable_timing(self, n_forwards: int):
        """Record stage events for the next ``n_forwards`` forwards (0 disables)."""
        _check("moe_layer_enable_timing", _get_lib().moe_layer_enable_timing(self._h, n_forwards))

    def stage_times(self) -> tuple[dict, int]:
        """Summed stage durations (ms) over the recorded forwards, and their count."""
        ms = (ctypes.c_float * len(STAGES))()
        n = ctypes.c_int32()
        _check("moe_layer_stage_times", _get_lib().moe_layer_stage_times(self._h, ms, ctypes.byref(n)))
        return dict(zip(STAGES, list(ms))), n.value

    def set_trace(self, buffer, n_ctas: int):
        """Profiling hook: per-CTA phase records of the fused decode kernel and the grouped
        GEMMs into a device buffer of n_ctas x 64 int64, n_ctas at least the SM count (None
        switches it off); the slots are listed with moe_layer_set_trace in the header. The
        kernels write into the buffer, so it must be a CUDA tensor of at least that size."""
        if buffer is not None:
            if not getattr(buffer, "is_cuda", False):
                raise TypeError("the trace buffer must be a CUDA tensor")
            if buffer.numel() * buffer.element_size() < int(n_ctas) * 64 * 8:
                raise ValueError(f"the trace buffer holds fewer than {n_ctas} x 64 int64")
        _check("moe_layer_set_trace", _get_lib().moe_layer_set_trace(self._h, _ptr(buffer), n_ctas))

    def launch_count(self) -> int:
        c = ctypes.c_int64()
        _check("moe_layer_launch_count", _get_lib().moe_layer_launch_count(self._h, ctypes.byref(c)))
        return c.value

    def status(self) -> int:
        return _get_lib().moe_layer_status(self._h)

    def set_wait_limit(self, ns: int):
        """Time limit (ns) of the kernels' waits on other CTAs (failure-handling hook)."""
        _check("moe_layer_set_wait_limit", _get_lib().moe_layer_set_wait_limit(self._h, int(ns)))

    def set_debug_checks(self, on: bool):
        """Check each forward's routing on the device (MOE_ERR_DEVICE_CHECK on a violation)."""
        _check("moe_layer_set_debug_checks", _get_lib().moe_layer_set_debug_checks(self._h, int(on)))

    def set_test_activation(self, identity: bool):
        """Test-only: h = gate * up instead of SiLU(gate) * up (exact-arithmetic cases)."""
        _check("moe_layer_set_test_activation", _get_lib().moe_layer_set_test_activation(self._h, int(identity)))

    def reset_status(self, stream=None):
        """Clear the sticky device status word."""
        _check("moe_layer_reset_status", _get_lib().moe_layer_reset_status(self._h, _stream(stream)))

    def nvfp4_act(self, T: int, stream=None) -> dict:
        """NVFP4 codes and E4M3 scales of the last forward's sorted routed x rows, and the
        amax of |x| (layers on the block-scaled FP4 path)."""
        rows, H = T * self.top_k, self.hidden
        r = {"codes": np.empty((rows, H // 2), np.uint8), "scales": np.empty((rows, H // 16), np.uint8),
             "amax": np.empty(1, np.float32)}
        _check("moe_layer_get_nvfp4_act", _get_lib().moe_layer_get_nvfp4_act(
            self._h, T, _ptr(r["codes"]), _ptr(r["scales"]), _ptr(r["amax"]), _stream(stream)))
        return r

    # ---------------------------------------------------------- HBM expert cache
    CACHE_STATS = ("hits", "misses", "prefetched", "prefetch_hits", "bytes_h2d", "evictions")

    def prefetch(self, x, stream=None):
        """Start loading the experts this layer's router predicts for x (device tensor)."""
        px = _act_ptr(x, self.hidden, self.act_dtype, True, "x")
        _check("moe_layer_prefetch", _get_lib().moe_layer_prefetch(self._h, px, x.shape[0], _stream(stream)))

    def cache_pin_hot(self, n: int):
        _check("moe_layer_cache_pin_hot", _get_lib().moe_layer_cache_pin_hot(self._h, int(n)))

    def cache_stats(self) -> dict:
        st = (ctypes.c_int64 * 6)()
        _check("moe_layer_cache_stats", _get_lib().moe_layer_cache_stats(self._h, st))
        return dict(zip(self.CACHE_STATS, list(st)))

    def cache_query(self) -> tuple[np.ndarray, np.ndarray]:
        """(slot of each routed expert or -1, pinned flags)."""
        slot = np.empty(self.n_experts, np.int32)
        pinned = np.empty(self.n_experts, np.int32)
        _check("moe_layer_cache_query", _get_lib().moe_layer_cache_query(self._h, _ptr(slot), _ptr(pinned)))
        return slot, pinned

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            _get_lib().moe_layer_destroy(self._h)
        self._h = _P()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
