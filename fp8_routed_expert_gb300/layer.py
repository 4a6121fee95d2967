"""Python face of the C ABI: argument marshalling around ``libfp8moe.so``.

Every step of the layer runs in the library's CUDA kernels; this module only
checks dtypes/shapes of torch tensors and passes their device pointers.
"""
from __future__ import annotations

import ctypes

import torch

from ._lib import C, MoEConfig, check, lib

PATHS = {"auto": C["MOE_PATH_AUTO"], "gemv": C["MOE_PATH_GEMV"], "gemm": C["MOE_PATH_GEMM"],
         "tcgemv": C["MOE_PATH_TCGEMV"]}
KERNELS = {name: C[f"MOE_K_{name.upper()}"] for name in
           ("router_logits", "router_select", "permute", "gate_up", "down", "combine", "act_quant",
            "route")}


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class MoELayer:
    """One routed-MoE layer context (workspace sized for max_tokens x max_top_k)."""

    def __init__(self, max_tokens: int, hidden: int, n_experts: int, inter: int, max_top_k: int,
                 device: int = 0):
        self.cfg = MoEConfig(max_tokens, hidden, n_experts, inter, max_top_k, device)
        self.device = device
        h = ctypes.c_void_p()
        check(lib().moe_init(ctypes.byref(h), ctypes.byref(self.cfg)), "moe_init")
        self._h = h

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().moe_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    def _check_weights(self, router_w, router_bias, w13, s13, w2, s2):
        c = self.cfg
        E, H, I = c.n_experts, c.hidden, c.inter
        want = [(router_w, torch.float32, (E, H)), (w13, torch.uint8, (E, 2 * I, H)),
                (s13, torch.float32, (E, 2 * I // 128, H // 128)), (w2, torch.uint8, (E, H, I)),
                (s2, torch.float32, (E, H // 128, I // 128))]
        if router_bias is not None:
            want.append((router_bias, torch.float32, (E,)))
        for t, dt, shape in want:
            if t.dtype != dt or tuple(t.shape) != shape or not t.is_contiguous() or not t.is_cuda:
                raise ValueError(f"expected contiguous cuda {dt} {shape}, got {t.dtype} {tuple(t.shape)}")

    def forward(self, x: torch.Tensor, router_w, router_bias, w13, s13, w2, s2, top_k: int,
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """x: bf16 [T, H] cuda.  Weights: see include/fp8moe.h.  Returns bf16 [T, H]."""
        if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != self.cfg.hidden or not x.is_contiguous():
            raise ValueError("x must be a contiguous bf16 [T, H] tensor")
        self._check_weights(router_w, router_bias, w13, s13, w2, s2)
        if out is None:
            out = torch.empty_like(x)
        rc = lib().moe_layer_forward(self._h, _ptr(x), x.shape[0], _ptr(router_w), _ptr(router_bias),
                                     _ptr(w13), _ptr(s13), _ptr(w2), _ptr(s2), top_k, _ptr(out),
                                     _stream_handle(stream))
        check(rc, "moe_layer_forward")
        return out

    def forward_nvfp4(self, x: torch.Tensor, router_w, router_bias, w13, sf13, g13, w2, sf2, g2,
                      top_k: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """The layer with FP4 (NVFP4) experts: w13 u8 [E, 2I, H/2], sf13 u8
        [E, 2I, H/16], g13 f32 [E]; w2 u8 [E, H, I/2], sf2 u8 [E, H, I/16],
        g2 f32 [E] (see include/fp8moe.h).  Returns bf16 [T, H]."""
        c = self.cfg
        E, H, I = c.n_experts, c.hidden, c.inter
        if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != H or not x.is_contiguous():
            raise ValueError("x must be a contiguous bf16 [T, H] tensor")
        want = [(router_w, torch.float32, (E, H)), (w13, torch.uint8, (E, 2 * I, H // 2)),
                (sf13, torch.uint8, (E, 2 * I, H // 16)), (g13, torch.float32, (E,)),
                (w2, torch.uint8, (E, H, I // 2)), (sf2, torch.uint8, (E, H, I // 16)),
                (g2, torch.float32, (E,))]
        if router_bias is not None:
            want.append((router_bias, torch.float32, (E,)))
        for t, dt, shape in want:
            if t.dtype != dt or tuple(t.shape) != shape or not t.is_contiguous() or not t.is_cuda:
                raise ValueError(f"expected contiguous cuda {dt} {shape}, got {t.dtype} {tuple(t.shape)}")
        if out is None:
            out = torch.empty_like(x)
        rc = lib().moe_layer_forward_nvfp4(self._h, _ptr(x), x.shape[0], _ptr(router_w),
                                           _ptr(router_bias), _ptr(w13), _ptr(sf13), _ptr(g13),
                                           _ptr(w2), _ptr(sf2), _ptr(g2), top_k, _ptr(out),
                                           _stream_handle(stream))
        check(rc, "moe_layer_forward_nvfp4")
        return out

    def forward_host(self, x_host: torch.Tensor, router_w, router_bias, w13, s13, w2, s2,
                     top_k: int, out_host: torch.Tensor, stream=None) -> torch.Tensor:
        """x_host, out_host: bf16 [T, H] CPU tensors (pinned for async copies)."""
        if x_host.is_cuda or out_host.is_cuda:
            raise ValueError("host entry point takes CPU tensors")
        self._check_weights(router_w, router_bias, w13, s13, w2, s2)
        rc = lib().moe_layer_forward_host(self._h, _ptr(x_host), x_host.shape[0], _ptr(router_w),
                                          _ptr(router_bias), _ptr(w13), _ptr(s13), _ptr(w2),
                                          _ptr(s2), top_k, _ptr(out_host), _stream_handle(stream))
        check(rc, "moe_layer_forward_host")
        return out_host

    def routing(self, T: int, k: int, stream=None) -> dict:
        """Routing of the last forward (T tokens, top-k) as torch tensors on the device."""
        dev = torch.device("cuda", self.device)
        E, P = self.cfg.n_experts, T * k
        r = dict(idx=torch.empty((T, k), dtype=torch.int32, device=dev),
                 wts=torch.empty((T, k), dtype=torch.float32, device=dev),
                 counts=torch.empty(E, dtype=torch.int32, device=dev),
                 offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                 perm=torch.empty(P, dtype=torch.int32, device=dev),
                 inv=torch.empty(P, dtype=torch.int32, device=dev))
        rc = lib().moe_get_routing(self._h, _ptr(r["idx"]), _ptr(r["wts"]), _ptr(r["counts"]),
                                   _ptr(r["offsets"]), _ptr(r["perm"]), _ptr(r["inv"]),
                                   _stream_handle(stream))
        check(rc, "moe_get_routing")
        return r

    def status(self) -> int:
        return lib().moe_status(self._h)

    def set_path(self, path: str) -> None:
        check(lib().moe_set_path(self._h, PATHS[path]), "moe_set_path")

    def resolved_path(self, T: int) -> str:
        """Name of the path a forward of T tokens takes ("gemv", "gemm" or "tcgemv")."""
        code = lib().moe_resolve_path(self._h, T)
        if code < 0:
            check(code, "moe_resolve_path")
        return {v: k for k, v in PATHS.items()}[code]

    def set_timing(self, kernels=()) -> None:
        """Time the named kernels (an iterable of KERNELS keys, or "all"); () turns timing off."""
        names = KERNELS if kernels == "all" else kernels
        mask = 0
        for n in names:
            mask |= 1 << KERNELS[n]
        check(lib().moe_set_timing(self._h, mask), "moe_set_timing")

    def launch_count(self) -> int:
        return int(lib().moe_launch_count(self._h))

    def kernel_time(self, kernel: str) -> tuple[float, int]:
        ms, n = ctypes.c_double(), ctypes.c_int64()
        check(lib().moe_kernel_time(self._h, KERNELS[kernel], ctypes.byref(ms), ctypes.byref(n)),
              "moe_kernel_time")
        return ms.value, n.value

    def debug_buffer(self, name: str, dtype: torch.dtype, shape, stream=None) -> torch.Tensor:
        """Copy of a workspace buffer of the last forward ('logits', 'h', 'y', 'x16')."""
        out = torch.empty(shape, dtype=dtype, device=torch.device("cuda", self.device))
        n = ctypes.c_int64()
        cap = out.numel() * out.element_size()
        check(lib().moe_debug_copy(self._h, name.encode(), _ptr(out), cap, ctypes.byref(n),
                                   _stream_handle(stream)), "moe_debug_copy")
        if cap > n.value:
            raise ValueError(f"buffer {name!r} holds {n.value} bytes, asked for {cap}")
        return out


CACHE_STATS = ("hits", "misses", "prefetched", "prefetch_used", "evictions", "bytes_copied")


class ExpertCache:
    """Experts kept in host memory with ``n_slots`` of them cached in device
    memory (see moe_cache_init in include/fp8moe.h).  ``w13_host`` /
    ``w2_host``: CPU uint8 tensors [E, 2I, H] / [E, H, I] that must stay alive
    and unchanged while the cache exists."""

    def __init__(self, layer: MoELayer, w13_host: torch.Tensor, w2_host: torch.Tensor, n_slots: int):
        c = layer.cfg
        E, H, I = c.n_experts, c.hidden, c.inter
        for t, shape in ((w13_host, (E, 2 * I, H)), (w2_host, (E, H, I))):
            if t.is_cuda or t.dtype != torch.uint8 or tuple(t.shape) != shape or not t.is_contiguous():
                raise ValueError(f"expected a contiguous CPU uint8 tensor {shape}")
        self.layer, self._keep = layer, (w13_host, w2_host)
        h = ctypes.c_void_p()
        check(lib().moe_cache_init(ctypes.byref(h), layer.handle, _ptr(w13_host), _ptr(w2_host),
                                   n_slots), "moe_cache_init")
        self._h = h

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().moe_cache_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, x: torch.Tensor, router_w, router_bias, s13, s2, top_k: int,
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty_like(x)
        rc = lib().moe_cache_forward(self._h, _ptr(x), x.shape[0], _ptr(router_w), _ptr(router_bias),
                                     _ptr(s13), _ptr(s2), top_k, _ptr(out), _stream_handle(stream))
        check(rc, "moe_cache_forward")
        return out

    def guess(self, x: torch.Tensor, router_w, router_bias, top_k: int, n_guess: int) -> list:
        buf = (ctypes.c_int32 * max(n_guess, 1))()
        n = lib().moe_cache_guess(self._h, _ptr(x), x.shape[0], _ptr(router_w), _ptr(router_bias),
                                  top_k, n_guess, buf)
        if n < 0:
            check(n, "moe_cache_guess")
        return list(buf[:n])

    def prefetch(self, experts) -> int:
        arr = (ctypes.c_int32 * max(len(experts), 1))(*experts)
        n = lib().moe_cache_prefetch(self._h, arr, len(experts))
        if n < 0:
            check(n, "moe_cache_prefetch")
        return n

    def stats(self) -> dict:
        buf = (ctypes.c_int64 * len(CACHE_STATS))()
        check(lib().moe_cache_stats(self._h, buf, len(CACHE_STATS)), "moe_cache_stats")
        return dict(zip(CACHE_STATS, buf))

    def resident(self) -> list:
        buf = (ctypes.c_int32 * self.layer.cfg.n_experts)()
        check(lib().moe_cache_resident(self._h, buf), "moe_cache_resident")
        return list(buf)
