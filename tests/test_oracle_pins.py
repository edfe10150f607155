"""The CPU oracle against facts fixed by the pages and by mathematics (no GPU)."""
import pytest

import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(orc, pin):
    pin(orc)


def test_pages_unit_totals():
    """Flat epilogue work-unit totals and concat shapes printed on the FusedQKV page."""
    shapes = {"qwen2.5-14b": (40, 8, 128, 5120), "qwen2.5-7b": (28, 4, 128, 3584)}
    seen = 0
    for row in pins.read_golden("pages_shapes.txt"):
        if row[0] == "units":
            nh, nkv, hd, _ = shapes[row[1]]
            assert (nh * hd) // 2 + (nkv * hd) // 2 + nkv * hd == int(row[2])
            seen += 1
        elif row[0] == "concat_shape":
            nh, nkv, hd, H = shapes[row[1]]
            assert (nh + 2 * nkv) * hd == int(row[2]) and H == int(row[3])
            seen += 1
    assert seen == 4
