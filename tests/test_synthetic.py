"""The seeded input generator (synthetic.py) on CPU: splitmix64 against its
published outputs, host (numpy) and device-side (PyTorch) generation bit for
bit -- the sampled parity checks recompute columns of full-size device inputs
on the host -- and the distributions' stated properties.
"""
import numpy as np
import pytest
import torch

import synthetic as S

KINDS = ("uniform", "normal", "uniform_bf16", "normal_bf16", "int")


def test_splitmix64_published_outputs():
    """S. Vigna's splitmix64: the first output from state 0, and the first five
    from seed 1234567 (the state advances by the golden-ratio increment)."""
    assert int(S.splitmix64_np(np.array([0], dtype=np.uint64))[0]) == 0xE220A8397B1DCDAF
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423,
            4593380528125082431, 16408922859458223821]
    states = np.array([(1234567 + k * 0x9E3779B97F4A7C15) % 2 ** 64 for k in range(5)], dtype=np.uint64)
    assert S.splitmix64_np(states).tolist() == want
    t = torch.tensor([S._signed(int(x)) for x in states], dtype=torch.int64)
    assert [v % 2 ** 64 for v in S.splitmix64_torch(t).tolist()] == want


def _bits(a):
    a = np.asarray(a)
    return a.view(np.uint16) if a.dtype == np.uint16 else a.view(np.uint8)


def _torch_to_np(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("start", [0, 2 ** 31 - 5, 2 ** 32 - 3, 2 ** 35 + 7])
def test_host_and_torch_generators_agree(kind, start):
    """Element indices past 2^31 and 2^32 included (the largest inputs the
    tests generate on the device)."""
    n = 4099
    for seed, rank, sigma in ((0, 0, 1.0), (5, 7, 1e-3), (3, 255, 1e-2)):
        dev = _torch_to_np(S.values_torch(kind, seed, rank, start, n, "cpu", sigma))
        host = S.values_np(kind, seed, rank, np.arange(start, start + n, dtype=np.uint64), sigma)
        assert dev.dtype == host.dtype
        assert np.array_equal(_bits(dev), _bits(host)), f"{kind} seed={seed} rank={rank} start={start}"


def test_pieces_compose():
    """Generating [0, n) in pieces gives the same values as in one go."""
    whole = S.values_torch("normal", 1, 2, 0, 1000, "cpu", 1e-3)
    parts = torch.cat([S.values_torch("normal", 1, 2, s, 250, "cpu", 1e-3) for s in range(0, 1000, 250)])
    assert torch.equal(whole.view(torch.int32), parts.view(torch.int32))


def test_distributions():
    idx = np.arange(200_000, dtype=np.uint64)
    u = S.values_np("uniform", 0, 1, idx)
    assert u.dtype == np.float32 and u.min() >= -1.0 and u.max() < 1.0
    assert np.all(u * np.float32(2 ** 23) == np.round(u * np.float32(2 ** 23)))  # multiples of 2^-23
    assert abs(float(u.mean())) < 0.01 and abs(float(u.var()) - 1 / 3) < 0.01
    x = S.values_np("normal", 0, 1, idx, 1e-3)
    assert abs(float(x.mean())) < 1e-5 and abs(float(x.std()) - 1e-3) < 2e-5   # sigma is the std dev
    k = S.values_np("int", 0, 1, idx)
    assert k.dtype == np.int32 and k.min() >= -(1 << 20) and k.max() <= (1 << 20)
    # ranks and seeds give different streams
    assert not np.array_equal(S.values_np("int", 0, 2, idx[:64]), k[:64])
    assert not np.array_equal(S.values_np("int", 1, 1, idx[:64]), k[:64])


def test_bf16_kinds_round_to_nearest_even():
    idx = np.arange(50_000, dtype=np.uint64)
    for kind, f32 in (("uniform_bf16", S.values_np("uniform", 4, 3, idx)),
                      ("normal_bf16", S.values_np("normal", 4, 3, idx, 1e-2))):
        bits = S.values_np(kind, 4, 3, idx, 1e-2)
        want = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(bits, want), kind
