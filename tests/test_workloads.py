"""The seeded input generators: Philox4x32-10 against its published
known-answer vectors, and the structure of the synthetic workloads."""
import numpy as np
import torch

from speculative_decoding_verification_41_gb300 import workloads as w

# Known-answer vectors of Philox4x32-10 published with the Random123 library of
# Salmon, Moraes, Dror and Shaw ("Parallel Random Numbers: As Easy as 1, 2, 3",
# SC'11): (counter, key) -> output.
PHILOX_KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


def test_philox_known_answers():
    for ctr, key, out in PHILOX_KAT:
        got = w.philox4x32_10(np.array([ctr], np.uint64), key)[0]
        assert tuple(int(x) for x in got) == out


def test_philox_stream_split_and_offsets():
    a = w.philox_words(7, 2, 37)
    b = w.philox_words(7, 2, 20, start=17)
    np.testing.assert_array_equal(a[17:], b)
    assert not np.array_equal(w.philox_words(7, 1, 8), w.philox_words(7, 2, 8))
    u = w.philox_uniforms(3, 2, 100000)
    assert u.dtype == np.float32 and u.min() >= 0 and u.max() < 1
    assert np.all((u.astype(np.float64) * 2 ** 24) % 1 == 0)      # on the 2^-24 grid
    assert abs(u.mean() - 0.5) < 0.005


def test_tiny_workload_is_deterministic():
    a, b = w.make_tiny(), w.make_tiny()
    for x, y in ((a.target_logits, b.target_logits), (a.draft_tokens, b.draft_tokens),
                 (a.uniforms, b.uniforms)):
        assert torch.equal(x, y)
    assert a.target_logits.shape == (4 * 5, 32) and a.draft_logits.shape == (4 * 4, 32)
    assert a.draft_tokens.min() >= 0 and a.draft_tokens.max() < 32


def test_ragged_workload_layout():
    vi = w.make_verify(5, 4, 300, torch.bfloat16, 0.7, rho=(0.6, 0.9), verify_len="uniform",
                       ragged=True, device="cpu")
    ell = vi.verify_len.numpy()
    assert ell.min() >= 1 and ell.max() <= 4
    np.testing.assert_array_equal(np.diff(vi.target_row_off.numpy()), ell + 1)
    np.testing.assert_array_equal(np.diff(vi.draft_row_off.numpy()), ell)
    assert vi.target_logits.shape[0] == int(vi.target_row_off[-1])
    assert vi.logit_bytes() == int((2 * ell + 1).sum()) * 300 * 2
    assert torch.isfinite(vi.target_logits.float()).all()


def test_step_time_profile():
    T = w.step_time_profile(5000)
    assert T[0] == 4.0 and abs(T[2048] - (4 + 0.006 * 2048)) < 1e-12
    assert abs(T[3000] - (4 + 0.006 * 2048 + 0.02 * 952)) < 1e-12
    c = w.make_confidences(512, 16)
    assert c.shape == (512, 16) and c.min() >= 0 and c.max() <= 1
    assert c[:, 0].mean() > c[:, 15].mean()
