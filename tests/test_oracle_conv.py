"""Pins for the causal depthwise conv1d oracle (page "PaddleNLP Kernel 算子库：CUDA
与 Triton 双实现的高性能 NLP GPU 算子实战指南", section 4.2, causal_conv1d_fn),
each against something other than the oracle itself: numpy.convolve per
channel, torch's silu, segment-by-segment convolution for seq_idx, and the
chained one-step update against the whole-sequence function.
"""
import numpy as np
import pytest
import torch

from oracle import conv1d

RTOL = 1e-13


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    den = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / den)


def _np_causal(row, taps, bias=0.0):
    """numpy.convolve of one row with the reversed taps, causal part."""
    return np.convolve(row, taps[::-1])[: len(row)] + bias


@pytest.mark.parametrize("width", [2, 3, 4])
def test_against_numpy_convolve(width):
    rng = np.random.default_rng(width)
    x, w, bias = rng.standard_normal((2, 5, 37)), rng.standard_normal((5, width)), rng.standard_normal(5)
    out = conv1d.causal_conv1d_ref(x, w, bias)
    for b in range(2):
        for d in range(5):
            assert _rel(out[b, d], _np_causal(x[b, d], w[d], bias[d])) < RTOL


def test_silu_and_swish_match_torch():
    rng = np.random.default_rng(3)
    x, w = rng.standard_normal((1, 4, 50)), rng.standard_normal((4, 4))
    lin = conv1d.causal_conv1d_ref(x, w)
    for act in ("silu", "swish"):
        got = conv1d.causal_conv1d_ref(x, w, activation=act)
        assert _rel(got, torch.nn.functional.silu(torch.from_numpy(lin)).numpy()) < 1e-15
    with pytest.raises(NotImplementedError):
        conv1d.causal_conv1d_ref(x, w, activation="relu")


def test_initial_states_extend_the_row():
    """With initial states the output is the convolution of [initial, x], its
    first width-1 outputs dropped; the final states are the last width-1
    entries of that row."""
    rng = np.random.default_rng(5)
    W = 4
    x, w, init = rng.standard_normal((2, 3, 20)), rng.standard_normal((3, W)), rng.standard_normal((2, 3, W - 1))
    out, fin = conv1d.causal_conv1d_ref(x, w, initial_states=init, return_final_states=True)
    for b in range(2):
        for d in range(3):
            row = np.concatenate([init[b, d], x[b, d]])
            assert _rel(out[b, d], _np_causal(row, w[d])[W - 1:]) < RTOL
            assert np.array_equal(fin[b, d], row[-(W - 1):])
    # a row shorter than width - 1 takes the rest of its final states from the initial states
    o2, f2 = conv1d.causal_conv1d_ref(x[:, :, :2], w, initial_states=init, return_final_states=True)
    assert np.array_equal(f2, np.concatenate([init[:, :, 2:], x[:, :, :2]], axis=2))


def test_seq_idx_restarts_each_sequence():
    """Packed sequences (seq_idx) equal separate convolutions of each segment."""
    rng = np.random.default_rng(7)
    W, L = 4, 30
    x, w, bias = rng.standard_normal((2, 3, L)), rng.standard_normal((3, W)), rng.standard_normal(3)
    cuts = [[0, 7, 8, 19, L], [0, 30]]
    seq = np.zeros((2, L), np.int32)
    for b, c in enumerate(cuts):
        for i in range(len(c) - 1):
            seq[b, c[i]:c[i + 1]] = i
    out = conv1d.causal_conv1d_ref(x, w, bias, seq_idx=seq)
    for b, c in enumerate(cuts):
        for d in range(3):
            ref = np.concatenate([_np_causal(x[b, d, c[i]:c[i + 1]], w[d], bias[d]) for i in range(len(c) - 1)])
            assert _rel(out[b, d], ref) < RTOL
    with pytest.raises(ValueError):
        conv1d.causal_conv1d_ref(x, w, seq_idx=seq, return_final_states=True)


def test_update_steps_chain_to_the_sequence():
    """l single-step updates from zero state reproduce the sequence output and
    end in the sequence's final states."""
    rng = np.random.default_rng(9)
    W = 3
    x, w, bias = rng.standard_normal((2, 4, 11)), rng.standard_normal((4, W)), rng.standard_normal(4)
    out, fin = conv1d.causal_conv1d_ref(x, w, bias, return_final_states=True, activation="silu")
    st = np.zeros((2, 4, W - 1))
    for t in range(11):
        o, st = conv1d.causal_conv1d_update_ref(x[:, :, t], st, w, bias, activation="silu")
        assert _rel(o, out[:, :, t]) < RTOL
    assert np.array_equal(st, fin)


def test_planted_mistakes_are_caught():
    """Taps in the wrong order, a shifted window, or a missing bias fail the
    numpy.convolve pin."""
    rng = np.random.default_rng(11)
    W = 4
    x, w, bias = rng.standard_normal(25), rng.standard_normal(W), 0.7
    ref = _np_causal(x, w, bias)
    ext = np.concatenate([np.zeros(W - 1), x])
    good = np.array([bias + sum(w[k] * ext[t + k] for k in range(W)) for t in range(25)])
    flipped = np.array([bias + sum(w[W - 1 - k] * ext[t + k] for k in range(W)) for t in range(25)])
    shifted = np.array([bias + sum(w[k] * np.concatenate([ext, [0.0]])[t + k + 1] for k in range(W)) for t in range(25)])
    nobias = good - bias
    assert _rel(good, ref) < RTOL
    for bad in (flipped, shifted, nobias):
        assert _rel(bad, ref) > 1e-3
