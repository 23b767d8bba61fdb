"""Per-tensor error-feedback state for stored weights ("fp4-train", API:
ErrorFeedback; Usage: the stored-weight loop, W = ef.qdq(name, W - lr * grad,
step=step)).

Each name owns one float32 residual of its weight's shape on the weight's
device, zero on first use; every call hands it to the library, which adds it
to the weight before quantizing and writes the new residual x + r - dq back
in place (Method: the residual is carried into the next quantization).  The
arithmetic is all the library's; this class only keeps the residuals.
"""
from __future__ import annotations

import torch

from . import nvfp4_qdq, nvfp4_quantize


class ErrorFeedback:
    """Residuals keyed by name.  ``stochastic`` selects stochastic rounding
    (keyed on (seed, step) and the element's index) over round-to-nearest;
    ``block`` is "1x16" or "16x16"."""

    def __init__(self, stochastic: bool = True, seed: int = 0, block: str = "1x16"):
        self.rounding = "sr" if stochastic else "rtn"
        self.seed = seed
        self.block = block
        self._res: dict[str, torch.Tensor] = {}

    def residual(self, name: str, like: torch.Tensor) -> torch.Tensor:
        """The residual of ``name``, created as zeros shaped like ``like``.  A
        weight of another shape or device than the residual's is refused
        rather than silently restarting its feedback."""
        r = self._res.get(name)
        if r is None:
            r = torch.zeros(like.shape, dtype=torch.float32, device=like.device)
            self._res[name] = r
        elif r.shape != like.shape or r.device != like.device:
            raise ValueError(f"ErrorFeedback: {name!r} holds a residual of shape {tuple(r.shape)} on "
                             f"{r.device}, not {tuple(like.shape)} on {like.device}")
        return r

    def qdq(self, name: str, w: torch.Tensor, step: int) -> torch.Tensor:
        """The bf16 value the stored weight takes: qdq(w + r), r updated."""
        return nvfp4_qdq(w, block=self.block, rounding=self.rounding, residual=self.residual(name, w),
                         seed=self.seed, step=step)["out"]

    def quantize(self, name: str, w: torch.Tensor, step: int) -> dict:
        """Codes and scale bytes of w + r, r updated (nvfp4_quantize's dict)."""
        return nvfp4_quantize(w, block=self.block, rounding=self.rounding, residual=self.residual(name, w),
                              seed=self.seed, step=step)

    def reset(self, name: str | None = None) -> None:
        """Drop one residual (or all of them): the next call starts from zero."""
        if name is None:
            self._res.clear()
        else:
            self._res.pop(name, None)

    def names(self) -> list[str]:
        return list(self._res)
