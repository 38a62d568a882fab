"""Size and seed of the seeded random-shape sweeps.

MOE_SWEEP_SCALE (default 1) multiplies the number of shapes of every sweep
and MOE_SWEEP_SEED (default 0) shifts every shape generator's seed, so that
a longer or a different sweep runs the same checks, e.g.

    MOE_SWEEP_SCALE=20 MOE_SWEEP_SEED=11 python -m pytest tests -m gpu -k random

The defaults give the sweeps the test suite always runs."""
import os

SCALE = max(1, int(os.environ.get("MOE_SWEEP_SCALE", "1")))
SEED = int(os.environ.get("MOE_SWEEP_SEED", "0"))


def count(n: int) -> int:
    return n * SCALE


def seed(base: int) -> int:
    return base + 1000003 * SEED
