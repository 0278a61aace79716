"""fp64 CPU oracle for the causal depthwise 1-D convolution.

TEST INFRASTRUCTURE ONLY: the tests and the bench's CPU-baseline leg use it;
the product path never does. It shares no code with the CUDA library.

The operator is ``causal_conv1d_fn(x, weight, bias=None, seq_idx=None,
initial_states=None, return_final_states=False, final_states_out=None,
activation=None)`` of the page "PaddleNLP Kernel 算子库：CUDA 与 Triton 双实现的
高性能 NLP GPU 算子实战指南", section 4.2: x (batch, dim, seqlen), a per-channel
(depthwise) kernel weight (dim, width), optional bias (dim,), optional
seq_idx (batch, seqlen) marking packed variable-length sequences (not together
with initial_states / return_final_states), optional initial_states
(batch, dim, width - 1) for decoding, activation None, "silu" or "swish".
The page gives the operands, not the formula; the plain reading taken here is
the causal convolution

    out[b, d, t] = act(bias[d] + sum_{k < width} weight[d, k] * x[b, d, t - (width - 1) + k])

where x at a position before 0 is the matching initial_states entry (else 0),
and, with seq_idx, a position whose seq_idx differs from position t's counts
as 0. silu = swish = v / (1 + e^-v). The final states are the last width - 1
inputs of each row (initial_states / zeros to the left when seqlen is shorter).

Written as explicit loops over the kernel taps on fp64 numpy arrays, in the
order of the definition.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        import torch
        return np.ascontiguousarray(x.detach().to("cpu", torch.float64).numpy())
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def causal_conv1d_ref(x, weight, bias=None, seq_idx=None, initial_states=None,
                      return_final_states=False, activation=None):
    """Returns out (b, d, l) fp64, and (out, final_states (b, d, width-1)) when
    return_final_states."""
    if activation not in (None, "silu", "swish"):
        raise NotImplementedError("activation must be None, silu or swish")
    if seq_idx is not None and (initial_states is not None or return_final_states):
        raise ValueError("seq_idx cannot be combined with initial_states / return_final_states")
    x, w = _f64(x), _f64(weight)
    b_, d_, l_ = x.shape
    W = w.shape[1]
    init = _f64(initial_states)
    # the row with its width - 1 left neighbours: [init or 0, x]
    left = init if init is not None else np.zeros((b_, d_, W - 1))
    ext = np.concatenate([left, x], axis=2)  # ext[..., j] = x[..., j - (W - 1)]
    sidx = None if seq_idx is None else np.asarray(seq_idx.cpu() if hasattr(seq_idx, "cpu") else seq_idx)
    out = np.zeros((b_, d_, l_))
    if bias is not None:
        out += _f64(bias)[None, :, None]
    t = np.arange(l_)
    for k in range(W):
        src = t - (W - 1) + k  # position read by tap k
        term = w[None, :, k:k + 1] * ext[:, :, src + (W - 1)]
        if sidx is not None:
            ok = (src >= 0)[None, :] & (sidx[:, np.clip(src, 0, None)] == sidx[:, t])
            term = term * ok[:, None, :]
        out += term
    if activation in ("silu", "swish"):
        out = out / (1.0 + np.exp(-out))
    if return_final_states:
        return out, ext[:, :, ext.shape[2] - (W - 1):].copy()
    return out


def causal_conv1d_update_ref(x, conv_state, weight, bias=None, activation=None):
    """One decode step: x (b, d) is the new input; conv_state (b, d, width - 1)
    holds the previous width - 1 inputs, oldest first. Returns
    (out (b, d), new conv_state) in fp64; the inputs are not modified."""
    if activation not in (None, "silu", "swish"):
        raise NotImplementedError("activation must be None, silu or swish")
    x, st, w = _f64(x), _f64(conv_state), _f64(weight)
    W = w.shape[1]
    window = np.concatenate([st, x[:, :, None]], axis=2)  # (b, d, W): oldest .. newest
    out = np.zeros(x.shape)
    if bias is not None:
        out += _f64(bias)[None, :]
    for k in range(W):
        out += w[None, :, k] * window[:, :, k]
    if activation in ("silu", "swish"):
        out = out / (1.0 + np.exp(-out))
    return out, window[:, :, 1:].copy()
