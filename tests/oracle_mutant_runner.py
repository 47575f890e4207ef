"""Runs every oracle pin against one build of the oracle library (a subprocess of
test_oracle_sensitivity).  Prints one line per pin, "FAILED <pin>" or "passed <pin>", flushed as
it goes, so that a planted mistake that crashes a later pin still shows the pins it failed before.

    python tests/oracle_mutant_runner.py <path of the oracle library>
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import numpy as np  # noqa: E402

import oracle_pins  # noqa: E402
from oracle.moe_oracle import Oracle  # noqa: E402


def main(path: str) -> int:
    O = Oracle(path)
    for pin in oracle_pins.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(O)
        except Exception as exc:  # an assertion, or an error the planted mistake causes
            print(f"FAILED {pin.__name__}: {type(exc).__name__}", flush=True)
        else:
            print(f"passed {pin.__name__}", flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1]))
