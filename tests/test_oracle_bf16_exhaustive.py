"""The oracle's float32 -> BF16 rounding over every one of the 2^32 float32 bit patterns.

The comparison rounds by the dropped-bits statement of nearest-even: keep the top 16 bits, and add one when the
dropped 16 bits are above half (0x8000), or exactly half with the kept value odd; NaNs give 0xFFFF (the pages'
code). The sampled pin in tests/pins.py checks the same rounding by float64 distances to both neighbours and
against PyTorch's conversion."""
import numpy as np


def test_bf16_every_float32_pattern(ora):
    chunk = 1 << 26
    base = np.arange(chunk, dtype=np.uint32)
    for start in range(0, 1 << 32, chunk):
        bits = base + np.uint32(start)
        got = ora.bf16_from_f32_bits(bits)
        kept = bits >> 16
        dropped = bits & 0xFFFF
        up = (dropped > 0x8000) | ((dropped == 0x8000) & ((kept & 1) == 1))
        want = (kept + up).astype(np.uint16)
        nan = (bits & 0x7FFFFFFF) > 0x7F800000
        want[nan] = 0xFFFF
        if not np.array_equal(got, want):
            bad = np.nonzero(got != want)[0][:5]
            raise AssertionError([(hex(bits[i]), hex(got[i]), hex(want[i])) for i in bad])
