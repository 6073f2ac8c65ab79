"""Pins of the causal depthwise convolution oracle (CPU)."""
import numpy as np
import pytest

from oracle import conv1d


def test_impulse_response_is_the_reversed_kernel():
    T, Cn, K = 12, 3, 4
    w = np.arange(1, Cn * K + 1, dtype=np.float64).reshape(Cn, K)
    u = np.zeros((T, Cn))
    u[5] = 1.0
    out, _ = conv1d.forward(u, w, silu=False)
    for j in range(K):
        assert np.array_equal(out[5 + j], w[:, K - 1 - j])
    assert not out[:5].any() and not out[5 + K:].any()


def test_identity_kernel_and_bias():
    rng = np.random.default_rng(0)
    u = rng.standard_normal((9, 5))
    w = np.zeros((5, 4))
    w[:, 3] = 1.0
    out, _ = conv1d.forward(u, w, bias=np.full(5, 0.5), silu=False)
    assert np.allclose(out, u + 0.5, rtol=0, atol=1e-15)
    out, pre = conv1d.forward(u, w, silu=True)
    assert np.allclose(out, u / (1 + np.exp(-u)), rtol=1e-15)


def test_matches_torch_grouped_conv1d():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    T, Cn, K = 40, 6, 4
    u = rng.standard_normal((T, Cn))
    w = rng.standard_normal((Cn, K))
    b = rng.standard_normal(Cn)
    ref = torch.nn.functional.conv1d(torch.tensor(u.T[None]), torch.tensor(w[:, None, :]), torch.tensor(b),
                                     padding=K - 1, groups=Cn)[0, :, :T].numpy().T
    out, pre = conv1d.forward(u, w, bias=b, silu=False)
    assert np.allclose(out, ref, rtol=1e-13, atol=1e-13)


def test_packed_equals_separate_sequences():
    rng = np.random.default_rng(2)
    cu = [0, 3, 3, 11, 20]
    u = rng.standard_normal((20, 4))
    w = rng.standard_normal((4, 4))
    b = rng.standard_normal(4)
    out, _ = conv1d.forward(u, w, bias=b, cu=cu)
    for s in range(len(cu) - 1):
        if cu[s + 1] > cu[s]:
            o, _ = conv1d.forward(u[cu[s]:cu[s + 1]], w, bias=b)
            assert np.array_equal(o, out[cu[s]:cu[s + 1]])


@pytest.mark.parametrize("silu", [True, False])
def test_gradients_by_central_differences(silu):
    rng = np.random.default_rng(3)
    cu = [0, 2, 9]
    u = rng.standard_normal((9, 3))
    w = rng.standard_normal((3, 4))
    b = rng.standard_normal(3)
    dout = rng.standard_normal((9, 3))
    du, dw, db = conv1d.backward(u, w, dout, bias=b, cu=cu, silu=silu)
    h = 1e-6

    def loss(u_, w_, b_):
        return float(np.sum(conv1d.forward(u_, w_, bias=b_, cu=cu, silu=silu)[0] * dout))

    for arr, grad, which in ((u, du, 0), (w, dw, 1), (b, db, 2)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            a1, a2 = arr.copy(), arr.copy()
            a1[idx] += h
            a2[idx] -= h
            args1, args2 = [u, w, b], [u, w, b]
            args1[which], args2[which] = a1, a2
            fd[idx] = (loss(*args1) - loss(*args2)) / (2 * h)
        assert np.allclose(grad, fd, rtol=1e-6, atol=1e-8)
