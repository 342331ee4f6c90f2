"""Pins for the oracle's GeLU (tanh form): torch's own tanh GeLU and its
autograd derivative in fp64, the closed forms at 0 and far out, and central
differences of the oracle's value."""
import numpy as np
import torch

import oracle


def test_gelu_matches_torch_tanh_gelu_and_its_derivative():
    x = torch.linspace(-8, 8, 4001, dtype=torch.float64, requires_grad=True)
    y = torch.nn.functional.gelu(x, approximate="tanh")
    y.sum().backward()
    assert np.max(np.abs(oracle.gelu(x.detach()) - y.detach().numpy())) < 1e-14
    assert np.max(np.abs(oracle.gelu_grad(x.detach()) - x.grad.numpy())) < 1e-13


def test_gelu_closed_forms():
    assert oracle.gelu(np.array([0.0]))[0] == 0.0
    assert oracle.gelu_grad(np.array([0.0]))[0] == 0.5
    big = np.array([30.0, -30.0])
    assert np.allclose(oracle.gelu(big), [30.0, 0.0], atol=1e-12)
    assert np.allclose(oracle.gelu_grad(big), [1.0, 0.0], atol=1e-12)


def test_gelu_grad_by_central_differences():
    x = np.linspace(-4, 4, 161)
    h = 1e-6
    fd = (oracle.gelu(x + h) - oracle.gelu(x - h)) / (2 * h)
    assert np.max(np.abs(fd - oracle.gelu_grad(x))) < 1e-8
