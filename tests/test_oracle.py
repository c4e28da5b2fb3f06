"""The CPU oracle against its pins (no GPU)."""
import pytest

import oracle_pins as P
from oracle import qlin_oracle as O


@pytest.mark.parametrize("name", [
    "hand_example", "file_layout", "forward_bruteforce", "quantize", "prologues",
    "closed_forms", "invariants", "stream_positions", "stream_bijection", "stream_positions_codebook", "stream_positions_rows", "bias", "moe",
    "codebook", "float_sanity",
])
def test_oracle_pin(name):
    getattr(P, "check_" + name)(O)
