"""Reader for the hand-derived fixtures under tests/golden/ (plain text, cited inside)."""

import os
import struct

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def e4m3_points():
    """[(float32 value, code, bf16_exact)] from e4m3_hand_derived.txt."""
    out = []
    with open(os.path.join(GOLDEN, "e4m3_hand_derived.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            _, bits, code, bf16, *_ = line.split()
            value = struct.unpack(">f", bytes.fromhex(bits[2:]))[0]
            out.append((value, int(code, 16), bf16 == "1"))
    return out
