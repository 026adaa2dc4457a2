"""Run every oracle pin against another build of the oracle source; print
one line per failing pin and exit 1 if any failed (used by
test_oracle_mutations.py in a subprocess, so that a broken copy cannot take
the test process down)."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import oracle  # noqa: E402
from pins import ALL_PINS  # noqa: E402


def main(so_path: str) -> int:
    L = oracle.load(so_path)
    failed = 0
    for pin in ALL_PINS:
        try:
            pin(L)
        except (AssertionError, ValueError) as e:
            print(f"FAILED {pin.__name__}: {type(e).__name__}: {e}", flush=True)
            failed += 1
    return 1 if failed else 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1]))
