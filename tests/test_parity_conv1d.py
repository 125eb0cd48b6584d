"""GPU parity of ssm_conv1d (causal depthwise Conv1D + SiLU) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_132_b300 as ssm

from _parity import assert_close, dev, host, io_dtype

pytestmark = pytest.mark.gpu


def _inputs(nb, L, D, K, seed, prev=False, bias=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((nb, L, D))
    w = rng.standard_normal((D, K)) / np.sqrt(K)
    b = rng.standard_normal(D) * 0.1 if bias else None
    xp = rng.standard_normal((nb, K - 1, D)) if prev else None
    return x, w, b, xp


def _round(a, io):
    """The values the kernel sees: inputs rounded to the I/O type."""
    if a is None:
        return None
    return host(dev(a, io_dtype(io)))


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("D", [64, 96, 1536, 37])          # vector rows, a ragged row width
@pytest.mark.parametrize("K", [4, 1, 3, 8])
def test_conv1d(io, D, K):
    nb, L = 3, 200                                         # 4 time blocks, ragged tail
    x, w, b, _ = _inputs(nb, L, D, K, seed=D * 10 + K)
    t = io_dtype(io)
    out = ssm.conv1d(dev(x, t), dev(w), dev(b))
    torch.cuda.synchronize()
    ref = oracle.conv1d(_round(x, io), w.astype(np.float32), None if b is None else
                        b.astype(np.float32))
    assert_close(host(out), ref, io, "conv1d+silu")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_conv1d_without_silu_or_bias(io):
    x, w, _, _ = _inputs(2, 70, 48, 4, seed=3, bias=False)
    t = io_dtype(io)
    out = ssm.conv1d(dev(x, t), dev(w), silu=False)
    torch.cuda.synchronize()
    ref = oracle.conv1d(_round(x, io), w.astype(np.float32), silu=False)
    assert_close(host(out), ref, io, "conv1d")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_conv1d_in_pieces_equals_whole(io):
    """A sequence run in two calls, the second fed the last K-1 inputs of the first,
    equals the single call (bit for bit: the same taps in the same order)."""
    nb, L, D, K = 2, 150, 64, 4
    x, w, b, _ = _inputs(nb, L, D, K, seed=9)
    t = io_dtype(io)
    xd, wd, bd_ = dev(x, t), dev(w), dev(b)
    whole = ssm.conv1d(xd, wd, bd_)
    cut = 77
    first = ssm.conv1d(xd[:, :cut].contiguous(), wd, bd_)
    second = ssm.conv1d(xd[:, cut:].contiguous(), wd, bd_,
                        x_prev=xd[:, cut - K + 1:cut].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([first, second], dim=1), whole)
    ref = oracle.conv1d(_round(x, io)[:, cut:], w.astype(np.float32), b.astype(np.float32),
                        x_prev=_round(x, io)[:, cut - K + 1:cut])
    assert_close(host(second), ref, io, "second piece")


def test_conv1d_empty_and_single_step():
    w = dev(np.ones((16, 4)))
    out = ssm.conv1d(torch.empty(2, 0, 16, device="cuda"), w)
    assert out.shape == (2, 0, 16)
    x, _, _, xp = _inputs(1, 1, 16, 4, seed=4, prev=True)
    got = ssm.conv1d(dev(x), w, x_prev=dev(xp))
    torch.cuda.synchronize()
    ref = oracle.conv1d(x, np.ones((16, 4)), x_prev=xp)
    assert_close(host(got), ref, "f32", "one step")


def test_conv1d_block_shape_full():
    """The 130M block's conv: batch 8, length 2048, d_inner 1536, K 4, bf16; every output
    against the oracle, with the channels (b, d) as rows."""
    nb, L, D, K = 8, 2048, 1536, 4
    x, w, b, _ = _inputs(nb, L, D, K, seed=11)
    t = torch.bfloat16
    out = host(ssm.conv1d(dev(x, t), dev(w), dev(b)))
    ref = oracle.conv1d(_round(x, "bf16"), w.astype(np.float32), b.astype(np.float32))
    assert_close(out, ref, "bf16", "conv1d block shape", row_axes=(0, 2))


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_conv1d_status_word_stays_clear(io):
    """With a status workspace the TMA-tiled kernel leaves SSM_OK there."""
    x, w, b, xp = _inputs(2, 300, 128, 4, seed=12, prev=True)
    t = io_dtype(io)
    ws = torch.full((256,), 7, dtype=torch.uint8, device="cuda")
    out = ssm.conv1d(dev(x, t), dev(w), dev(b), x_prev=dev(xp, t), workspace=ws)
    torch.cuda.synchronize()
    assert ssm.read_device_status(ws) == 0
    ref = oracle.conv1d(_round(x, io), w.astype(np.float32), b.astype(np.float32),
                        x_prev=_round(xp, io))
    assert_close(host(out), ref, io, "conv1d with carried window")
