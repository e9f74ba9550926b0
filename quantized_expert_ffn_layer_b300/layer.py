"""Device-resident weights + workspace around the libftmoe calls (marshalling only)."""
from __future__ import annotations

import numpy as np
import torch

from . import ftmoe as F


def upload_tiles(qtype: str, canon: np.ndarray, E: int, N: int, K: int, device, stream=None, ts=None):
    """Canonical block bytes (host numpy uint8 [E, N, K/bs, blk]) -> device tiles via
    ftmoe_repack; NVFP4 also takes the E fp32 tensor scales (appended to the canonical
    buffer, as ftmoe_repack reads them)."""
    raw = np.ascontiguousarray(canon).reshape(-1)
    if ts is not None:
        raw = np.concatenate([raw, np.ascontiguousarray(ts, dtype="<f4").view(np.uint8)])
    src = torch.from_numpy(raw).to(device)
    tiles = torch.empty(F.ftmoe_tiled_bytes(qtype, E, N, K), dtype=torch.uint8, device=device)
    F.ftmoe_repack(qtype, src, tiles, E, N, K, stream)
    torch.cuda.current_stream(device).synchronize() if stream is None else stream.synchronize()
    del src
    return tiles


class MoELayer:
    """One MoE layer's weights on the device in the kernels' tiled layout."""

    def __init__(self, qtype, E, H, I, w13, w2, shared_w13=None, shared_w2=None, device="cuda",
                 ts=None):
        """ts: NVFP4's tensor scales {"w13": [E], "w2": [E], "shared_w13": [1], "shared_w2": [1]}."""
        self.qtype, self.E, self.H, self.I = qtype, E, H, I
        self.device = torch.device(device)
        t = ts or {}
        self.w13 = upload_tiles(qtype, w13, E, 2 * I, H, self.device, ts=t.get("w13"))
        self.w2 = upload_tiles(qtype, w2, E, H, I, self.device, ts=t.get("w2"))
        self.shared = shared_w13 is not None
        self.sw13 = self.sw2 = None
        if self.shared:
            self.sw13 = upload_tiles(qtype, shared_w13, 1, 2 * I, H, self.device, ts=t.get("shared_w13"))
            self.sw2 = upload_tiles(qtype, shared_w2, 1, H, I, self.device, ts=t.get("shared_w2"))
        self.weights = F.make_weights(qtype, E, H, I, self.w13, self.w2, None, self.sw13, self.sw2)
        self._ws = None

    def workspace(self, T, k):
        n = F.ftmoe_layer_workspace_bytes(T, k, self.E, self.H, self.I, self.shared)
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty(max(n, 256), dtype=torch.uint8, device=self.device)
        return self._ws

    def capture(self, fn):
        """Records fn() (calls of this layer and any stream-ordered copies around them) into a
        CUDA graph and returns it: graph.replay() reruns every kernel and copy of fn on the
        same buffers with one launch.  fn runs once first, outside the capture, so that the
        kernels' one-time settings are made before recording."""
        s = torch.cuda.Stream(self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            fn()
        torch.cuda.current_stream(self.device).wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fn()
        return g

    def forward(self, logits, x_bf16, k, out=None, ids_out=None, w_out=None, stream=None):
        """logits fp32 [T, E], x bf16 [T, H] (device) -> out bf16 [T, H]."""
        T = x_bf16.shape[0]
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.bfloat16, device=self.device)
        ws = self.workspace(T, k)
        F.ftmoe_layer(self.weights, logits, x_bf16, T, k, out, ids_out, w_out, ws, ws.numel(), stream)
        return out
