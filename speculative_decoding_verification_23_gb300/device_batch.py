"""Moves a ``workload.Batch`` to the GPU in the layout the C ABI expects
(argument marshalling only: host -> device copies, dtype casts of the
inputs, no arithmetic of the method)."""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np


@dataclasses.dataclass
class DeviceBatch:
    B: int
    V: int
    max_k: int
    target: object
    draft: object
    cu_draft: object
    draft_tokens: object
    cu_hist: object
    hist: object
    temperature: object
    rep_penalty: object
    top_p: Optional[object]
    tv_budget: object
    uniforms: object

    def args(self, *, flags: int = 0, with_top_p: Optional[bool] = None, with_penalty: bool = True):
        from . import make_args

        use_tp = self.top_p is not None if with_top_p is None else with_top_p
        return make_args(target=self.target, draft=self.draft, cu_draft=self.cu_draft,
                         draft_tokens=self.draft_tokens, V=self.V, cu_hist=self.cu_hist, hist=self.hist,
                         temperature=self.temperature, rep_penalty=self.rep_penalty if with_penalty else None,
                         top_p=self.top_p if use_tp else None, tv_budget=self.tv_budget,
                         uniforms=self.uniforms, max_k=self.max_k, flags=flags)


def to_device(batch, device="cuda", *, pin: bool = False) -> DeviceBatch:
    import torch

    def f32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)

    def logits(a):
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
        if batch.dtype == "bf16":
            t = t.to(torch.bfloat16)       # exact: the values are bf16-representable
        return t.to(device)

    draft = batch.draft if batch.draft.shape[0] > 0 else np.zeros((1, batch.ld), np.float32)
    tokens = batch.draft_tokens if batch.draft_tokens.size else np.zeros(0, np.int32)
    hist = batch.hist if batch.hist.size else np.zeros(1, np.int32)
    top_p = None if np.all(batch.top_p >= 1.0) else f32(batch.top_p)
    return DeviceBatch(B=batch.B, V=batch.V, max_k=max(batch.max_k, 0), target=logits(batch.target),
                       draft=logits(draft), cu_draft=i32(batch.cu_draft), draft_tokens=i32(tokens),
                       cu_hist=i32(batch.cu_hist), hist=i32(hist), temperature=f32(batch.temperature),
                       rep_penalty=f32(batch.rep_penalty), top_p=top_p, tv_budget=f32(batch.tv_budget),
                       uniforms=f32(batch.uniforms))
