"""The seeded input generator: deterministic, distribution as stated, and independent
of the device (the GPU check lives in test_gpu_parity.py)."""
import numpy as np
import torch

from gqa_decoder_forward_gb300 import synth


def test_deterministic_and_seed_dependent():
    a = synth.normal_bf16(1, 3, (1000,), 0.02)
    b = synth.normal_bf16(1, 3, (1000,), 0.02)
    c = synth.normal_bf16(2, 3, (1000,), 0.02)
    d = synth.normal_bf16(1, 4, (1000,), 0.02)
    assert torch.equal(a, b)
    assert not torch.equal(a, c) and not torch.equal(a, d)


def test_normal_moments_and_bounds():
    x = synth.normal_bf16(11, 0, (1 << 20,), 0.02).float()
    assert abs(x.mean().item()) < 2e-4
    assert abs(x.std().item() - 0.02) < 4e-4
    assert x.abs().max().item() <= 0.02 * 3.47
    n = synth.normal_bf16(11, 1, (1 << 16,), 0.1, mean=1.0).float()
    assert abs(n.mean().item() - 1.0) < 2e-3 and abs(n.std().item() - 0.1) < 3e-3


def test_chunking_does_not_change_values(monkeypatch):
    a = synth.normal_bf16(5, 9, (3000,), 1.0)
    monkeypatch.setattr(synth, "_CHUNK", 7)
    b = synth.normal_bf16(5, 9, (3000,), 1.0)
    assert torch.equal(a, b)


def test_uniform_ids_cover_vocab():
    ids = synth.uniform_ids(2, 200000, 4096)
    assert ids.dtype == torch.int32
    assert ids.min().item() == 0 and ids.max().item() == 4095
    counts = np.bincount(ids.numpy(), minlength=4096)
    assert counts.min() > 10


def test_bits_roundtrip():
    t = synth.normal_bf16(1, 1, (5, 7), 1.0)
    b = synth.bits(t)
    assert b.dtype == np.uint16 and b.shape == (5, 7)
    back = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16)
    assert torch.equal(back, t)
