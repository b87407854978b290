"""Pins for the oracle's output projection y = o . W_O ("vLLM Fork with
focus on GB10 Homelabs", "Roadmap": fused attention + W_O GEMV), against
closed forms and an independent library matmul: the identity, a single
nonzero weight (catches a transposed operand or a wrong head order), a
known bf16 weight value (catches a wrong decode of W), torch fp64."""
import numpy as np
import torch

import oracle


def bits(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_identity_returns_the_flattened_output():
    o = np.random.default_rng(0).standard_normal((3, 1, 4, 8))
    y = oracle.wo_project(o, bits(np.eye(32)))
    assert np.array_equal(y, o.reshape(3, 32))


def test_single_weight_selects_one_head_element():
    rng = np.random.default_rng(1)
    o = rng.standard_normal((2, 1, 6, 16))     # k = head * 16 + d
    W = np.zeros((96, 40), np.float32)
    W[3 * 16 + 5, 17] = 1.0                     # head 3, d 5 -> column 17
    y = oracle.wo_project(o, bits(W))
    assert np.array_equal(y[:, 17], o[:, 0, 3, 5])
    assert not np.delete(y, 17, axis=1).any()


def test_known_bf16_weight_value():
    o = np.random.default_rng(2).standard_normal((2, 1, 2, 4))
    W = np.zeros((8, 3), np.uint16)
    W[:, 1] = 0x3FC0                            # bf16 1.5
    W[:, 2] = 0xC080                            # bf16 -4.0
    y = oracle.wo_project(o, W)
    s = o.reshape(2, 8).sum(axis=1)
    np.testing.assert_allclose(y[:, 1], 1.5 * s, rtol=1e-13)
    np.testing.assert_allclose(y[:, 2], -4.0 * s, rtol=1e-13)
    assert not y[:, 0].any()


def test_matches_torch_fp64_matmul():
    g = torch.Generator().manual_seed(3)
    o = torch.randn(5, 1, 8, 32, generator=g, dtype=torch.float64)
    W = (torch.randn(256, 64, generator=g) / 16).to(torch.bfloat16)
    y = oracle.wo_project(o.numpy(), W.view(torch.int16).numpy().view(np.uint16))
    ref = (o.reshape(5, 256) @ W.double()).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-14)
