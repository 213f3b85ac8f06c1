"""Oracle values for sampled tokens of a full-size layer.

The layer's output row of token t depends only on t's own routed rows once
the activation's per-tensor scale and the routing are fixed, so the oracle
can check a sample of tokens at sizes where running it on every token would
take hours.  For each sampled (token, slot) pair this module computes,
strictly through oracle functions: the float32 SwiGLU row, its
requantisation (codes and block scales), the bf16 down-projection row, and
per token the bf16 layer output summed in slot order.

Cost is dominated by quantising each involved expert's weight matrices with
the oracle (tens of millions of elements each); experts are independent, so
they run on a thread pool (numpy releases the interpreter lock inside its
array loops), and each matrix is quantised in row chunks so a worker's
temporaries stay small.  Quantisation is defined row by row (a row's codes
and block scales depend only on the row and the matrix's per-tensor scale),
so chunking changes nothing.

This is test code: it imports the oracle, never the CUDA library.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from oracle import nvfp4_moe_oracle as O

ROW_CHUNK = 1024


def _matrix(w, e):
    """Expert e of a [E, N, K] weight stack (torch, any device, or numpy) as float32 numpy."""
    m = w[int(e)]
    if hasattr(m, "cpu"):
        m = m.cpu().float().numpy()
    return np.asarray(m, dtype=np.float32)


def _times_weights_t(xd, a, fmt):
    """xd [n, K] float64 times the transposed oracle quantisation of the
    weight matrix a [N, K] (float32): returns [n, N] float64."""
    out = np.empty((xd.shape[0], a.shape[0]), dtype=np.float64)
    g = None if fmt == "mxfp4" else O.global_scale(a)
    for r0 in range(0, a.shape[0], ROW_CHUNK):
        blk = a[r0:r0 + ROW_CHUNK]
        if fmt == "mxfp4":
            wd = O.dequantize_mxfp4(*O.quantize_mxfp4(blk))
        else:
            wd = O.dequantize_nvfp4(*O.quantize_nvfp4(blk, g), g)
        out[:, r0:r0 + ROW_CHUNK] = xd @ wd.T
    return out


def expert_rows(w_gu, w_d, e, xd, I, fmt="nvfp4", s_h=None):
    """Oracle rows of expert e for dequantised activation rows xd [n, H]:
    (h float32 [n, I], h codes [n, I], h block scales, y bf16-rounded float64 [n, H])."""
    gu = _times_weights_t(xd, _matrix(w_gu, e), fmt)
    h = O.swiglu(gu, I).astype(np.float32)
    if fmt == "mxfp4":
        hq, hs = O.quantize_mxfp4(h)
        hd = O.dequantize_mxfp4(hq, hs)
    else:
        hq, hs = O.quantize_nvfp4(h, np.float32(s_h))
        hd = O.dequantize_nvfp4(hq, hs, np.float32(s_h))
    y = O.round_to_bf16(_times_weights_t(hd, _matrix(w_d, e), fmt))
    return h, O.unpack_codes(hq), hs, y


def default_threads():
    return max(1, min(os.cpu_count() or 1, 16))


class TokenSample:
    """Oracle values of the sampled tokens `tokens` of a layer.

    x32: float32 [T, H] activations (bf16 values); idx, wts: the oracle's
    routing of the whole batch; w_gu [E, 2I, H], w_d [E, H, I]: the bf16
    master weights (torch tensors, any device); s_x: the activation's
    per-tensor scale (NVFP4); s_h: the SwiGLU output's static scale.
    Attributes, per pair (token tokens[i], slot j) in row-major order:
    pairs [n, 2] (token, slot), experts [n], h, h_codes, h_scales, y; and
    out [len(tokens), H]: the bf16 layer output of each sampled token."""

    def __init__(self, tokens, x32, idx, wts, w_gu, w_d, fmt="nvfp4", s_x=None, s_h=None, threads=None):
        self.tokens = np.asarray(tokens, dtype=np.int64)
        T, k = idx.shape
        H = x32.shape[1]
        I = w_d.shape[2]
        self.pairs = np.stack(np.meshgrid(self.tokens, np.arange(k), indexing="ij"), -1).reshape(-1, 2)
        self.experts = idx[self.pairs[:, 0], self.pairs[:, 1]].astype(np.int64)
        if fmt == "mxfp4":
            xd = O.dequantize_mxfp4(*O.quantize_mxfp4(x32[self.tokens]))
        else:
            xd = O.dequantize_nvfp4(*O.quantize_nvfp4(x32[self.tokens], s_x), s_x)
        row_of_token = {int(t): i for i, t in enumerate(self.tokens)}
        n = len(self.pairs)
        blk = 32 if fmt == "mxfp4" else 16
        self.h = np.empty((n, I), np.float32)
        self.h_codes = np.empty((n, I), np.uint8)
        self.h_scales = np.empty((n, I // blk), np.uint8)
        self.y = np.empty((n, H), np.float64)

        def one(e):
            sel = np.nonzero(self.experts == e)[0]
            rows = np.array([row_of_token[int(t)] for t in self.pairs[sel, 0]])
            return sel, expert_rows(w_gu, w_d, e, xd[rows], I, fmt, s_h)

        with ThreadPoolExecutor(threads or default_threads()) as ex:
            for sel, (h, hc, hs, y) in ex.map(one, np.unique(self.experts)):
                self.h[sel], self.h_codes[sel], self.h_scales[sel], self.y[sel] = h, hc, hs, y
        acc = np.zeros((len(self.tokens), H), np.float64)
        wp = wts[self.pairs[:, 0], self.pairs[:, 1]].astype(np.float64).reshape(len(self.tokens), k)
        yk = self.y.reshape(len(self.tokens), k, H)
        for j in range(k):                        # slot order (reading R7)
            acc += wp[:, j:j + 1] * yk[:, j]
        self.out = O.round_to_bf16(acc)

    def flat_ids(self, k):
        """Flat routed-row ids t*k + j of the pairs."""
        return self.pairs[:, 0] * k + self.pairs[:, 1]
