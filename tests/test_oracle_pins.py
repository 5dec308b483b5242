"""The oracle against its pins (see tests/pins.py for what each pin holds it to)."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(ora, pin):
    pin(ora)


def test_golden_derivation_rejects_a_wrong_line(tmp_path, monkeypatch):
    """The hand-worked derivations are checked line by line: one flipped bit in one result is refused."""
    import golden_steps
    text = open(golden_steps.os.path.join(golden_steps.GOLDEN, "adamw_op_order.txt")).read()
    assert golden_steps.read_cases(), "no derivations"
    target = "op m1 = m + cdm = 0x"
    i = text.index(target) + len(target)
    bad = text[:i] + format(int(text[i:i + 8], 16) ^ 1, "08x") + text[i + 8:]
    (tmp_path / "adamw_op_order.txt").write_text(bad)
    monkeypatch.setattr(golden_steps, "GOLDEN", str(tmp_path))
    with pytest.raises(AssertionError, match="m1 = m"):
        golden_steps.read_cases()
