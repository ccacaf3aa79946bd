"""A quantized linear layer on the library.

The Humming README's usage example drives a layer object: construct it with
the output and input sizes and a weight configuration, load the quantized
tensors, transform them for the device, then call it on activations.  This
class offers the same sequence on top of the C ABI: ``load`` takes the
standard-format tensors (``include/hq.h``), ``transform`` runs
``hq_transform``, and a call runs ``hq_gemm`` on the current torch stream.
Marshalling only: torch provides device memory, every computation runs in
the library's kernels.
"""
from __future__ import annotations

import torch

from . import (hq_gemm, hq_gemm_workspace_size, hq_status_read, hq_transform, hq_transform_size,
               hq_workspace_init, make_desc)

_ELEM = {"bf16": 2, "fp16": 2, "fp8": 1}


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


class QuantLinear:
    """Y = a(X) . dequant(W)^T for one dense quantized weight W [n, k].

    The layer keeps one workspace (status word and split-K counters) for all
    its calls, so calls of one layer must be ordered on one stream (or by
    events); calls that overlap on the GPU race on it.  ``status()`` reads
    the workspace's device status word and, when a device-side error was
    recorded there, clears the whole workspace so that later calls start
    from zeroed counters.
    """

    def __init__(self, n: int, k: int, wtype: str, stype: str, group_k: int = 128, group_n: int = 1,
                 signed_codes: bool = True, has_zeros: bool = False, device="cuda"):
        self.n, self.k = n, k
        self.wtype, self.stype = wtype, stype
        self.group_k, self.group_n = group_k, group_n
        self.signed_codes, self.has_zeros = signed_codes, has_zeros
        self.device = torch.device(device)
        self._std = None
        self.wt = None
        self._ws = None
        # validates the configuration (raises HQError for an invalid one)
        self.transformed_bytes = hq_transform_size(self._desc())

    def _desc(self, codes=None, scales=None, zeros=None):
        return make_desc(self.wtype, self.stype, self.n, self.k, 1, self.group_k, self.group_n, self.signed_codes,
                         self.has_zeros, codes, scales, zeros)

    def standard_bytes(self) -> dict:
        """Byte sizes of the standard-format tensors this configuration takes."""
        n, k, g = self.n, self.k, self.group_k
        groups = 1 if g == 0 else k // g
        if self.wtype == "int4":
            codes, scales, zeros = n * _cdiv(k, 2), 2 * n * groups, n * _cdiv(groups, 2)
        elif self.wtype == "int6":
            codes, scales, zeros = n * 3 * k // 4, 2 * n * groups, n * 3 * _cdiv(groups, 4)
        elif self.wtype == "mxfp4":
            codes, scales, zeros = n * k // 2, n * k // 32, 0
        else:  # fp8 blocks
            codes, scales, zeros = n * k, 4 * _cdiv(n, 128) * _cdiv(k, 128), 0
        return {"codes": codes, "scales": scales, "zeros": zeros if self.has_zeros else 0}

    def load(self, codes: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor | None = None) -> "QuantLinear":
        """Take the standard-format tensors (contiguous, on this layer's device)."""
        want = self.standard_bytes()
        got = {"codes": codes, "scales": scales, "zeros": zeros}
        for name, t in got.items():
            if want[name] == 0:
                if t is not None:
                    raise ValueError(f"{name}: this configuration takes none")
                continue
            if t is None:
                raise ValueError(f"{name}: required")
            if not t.is_contiguous():
                raise ValueError(f"{name}: must be contiguous")
            if t.numel() * t.element_size() != want[name]:
                raise ValueError(f"{name}: {t.numel() * t.element_size()} bytes, the configuration takes {want[name]}")
        self._std = (codes, scales, zeros)
        return self

    def transform(self) -> "QuantLinear":
        """Repack the loaded tensors into the device tile layout (hq_transform)."""
        if self._std is None:
            raise RuntimeError("load() first")
        codes, scales, zeros = self._std
        buf = torch.empty(self.transformed_bytes + 256, dtype=torch.uint8, device=self.device)
        off = (-buf.data_ptr()) % 256                       # the transformed buffer is 256-byte aligned
        self.wt = buf[off:off + self.transformed_bytes]
        hq_transform(self._desc(codes, scales, zeros), self.wt, self.transformed_bytes,
                     torch.cuda.current_stream(self.device))
        self._std = None                                    # the standard tensors are no longer needed
        return self

    def __call__(self, x: torch.Tensor, x_scales: torch.Tensor | None = None, flags: int = 0) -> torch.Tensor:
        """x [m, k]: bf16 / fp16, or e4m3 bytes (uint8 or float8_e4m3fn) with float32 x_scales
        [m, ceil(k/128)].  Returns Y [m, n], bf16 (fp16 for fp16 activations)."""
        if self.wt is None:
            raise RuntimeError("transform() first")
        if x.dim() != 2 or x.shape[1] != self.k:
            raise ValueError(f"x must be [m, {self.k}]")
        if x.dtype == torch.bfloat16:
            atype = "bf16"
        elif x.dtype == torch.float16:
            atype = "fp16"
        elif x.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
            atype = "fp8"
            x = x.view(torch.uint8)
        else:
            raise ValueError(f"unsupported activation dtype {x.dtype}")
        m = x.shape[0]
        esz = _ELEM[atype]
        # rows 16-byte aligned, as the tensor copies need (copy into a padded buffer otherwise)
        if x.stride(1) != 1 or (x.stride(0) * esz) % 16 or x.data_ptr() % 16:
            ldx = _cdiv(self.k * esz, 16) * 16 // esz
            xp = torch.zeros((m, ldx), dtype=x.dtype, device=x.device)
            xp[:, :self.k] = x
            x = xp
        ldx = x.stride(0)
        ldy = _cdiv(self.n, 8) * 8
        y = torch.empty((m, ldy), dtype=torch.float16 if atype == "fp16" else torch.bfloat16, device=x.device)
        if m == 0:
            return y[:, :self.n]
        desc = self._desc()
        need = hq_gemm_workspace_size(desc, m, atype)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=x.device)   # zero = initialised
        if atype == "fp8":
            if x_scales is None or x_scales.dtype != torch.float32 or not x_scales.is_contiguous():
                raise ValueError("fp8 activations need contiguous float32 x_scales [m, ceil(k/128)]")
        hq_gemm(desc, self.wt, m, atype, x, ldx, x_scales if atype == "fp8" else None, y, ldy, self._ws,
                self._ws.numel(), flags, torch.cuda.current_stream(x.device))
        return y[:, :self.n]

    def status(self, clear: bool = True) -> int:
        """Synchronise the current stream and return the device status of the
        last calls (0 = HQ_OK).  With ``clear``, a non-zero status resets the
        workspace (status word and split-K counters) on the current stream."""
        if self._ws is None:
            return 0
        s = torch.cuda.current_stream(self._ws.device)
        st = hq_status_read(self._ws, clear=False, stream=s)
        if st != 0 and clear:
            hq_workspace_init(self._ws, self._ws.numel(), s)
        return st
