"""The CPU oracle against its pins (closed forms, library routines, the pages' numbers)."""
import pytest

from pins import PINS


@pytest.mark.parametrize("name", sorted(PINS))
def test_pin(ora, name):
    PINS[name](ora)


def test_oracle_digest_unchanged():
    """The oracle's outputs on fixed inputs match the committed digest."""
    import json
    import os
    from golden import make_oracle_digest as mk
    want = json.load(open(mk.OUT))
    got = mk.run()
    for k, v in got.items():
        assert want[k] == v, "oracle output changed for %s" % k
