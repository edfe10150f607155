"""The seeded input generator (no GPU): published SplitMix64 outputs, normal statistics,
per-row keying that makes separate wq/wk/wv blocks equal the concat rows, determinism."""
import numpy as np

from qkv_rope_kv_gb300 import synth


def test_splitmix64_published_sequence():
    # First outputs of SplitMix64 started from state 0 (Vigna's reference splitmix64.c).
    assert synth.splitmix64(0, 1) == 0xE220A8397B1DCDAF
    assert synth.splitmix64(0, 2) == 0x6E789E6AA1B965F4
    assert synth.splitmix64(0, 3) == 0x06C45D188009454F


def test_normal_statistics():
    z = synth.normal_f32(0, 99, 0, 0, 400000, 1.0).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    assert abs(np.mean(z ** 3)) < 0.03 and abs(np.mean(z ** 4) - 3.0) < 0.05
    w = synth.weight_rows(0, 0, 0, 64, 1024, "f32").astype(np.float64)
    assert abs(w.std() - synth.W_SIGMA) < 0.02 * synth.W_SIGMA


def test_row_keying_makes_blocks_equal_concat():
    H, R = 96, 40
    full = synth.weight_rows(0, 3, 0, R, H, "bf16")
    assert np.array_equal(full[10:25], synth.weight_rows(0, 3, 10, 15, H, "bf16"))
    f32 = synth.weight_rows(0, 3, 0, R, H, "f32")
    # bf16 is the RN-even rounding of the f32 value
    b = f32.view(np.uint32)
    rne = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)
    assert np.array_equal(full, rne)


def test_streams_are_distinct_and_deterministic():
    a = synth.hidden(0, 1, 17, 512)
    assert np.array_equal(a, synth.hidden(0, 1, 17, 512))
    for other in (synth.hidden(0, 2, 17, 512), synth.hidden(0, 1, 18, 512), synth.hidden(1, 1, 17, 512)):
        assert not np.array_equal(a, other)
