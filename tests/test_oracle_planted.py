"""The pins of tests/test_oracle_pins.py catch plausible mistakes: the oracle
is rebuilt with one planted mistake at a time (ORC_PLANT_* in oracle.c, never
defined otherwise) and the pin suite must fail for each."""
import os
import subprocess
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
PLANTS = ["ORC_PLANT_SLOT_OFFSET", "ORC_PLANT_GQA_MODULO", "ORC_PLANT_NO_SCALE",
          "ORC_PLANT_CAUSAL_OFF_BY_ONE", "ORC_PLANT_NO_RESCALE", "ORC_PLANT_KEEP_PADDING",
          "ORC_PLANT_V_REVERSED", "ORC_PLANT_ROUND_TRUNC", "ORC_PLANT_NORM_SUM",
          "ORC_PLANT_EPS_OUTSIDE", "ORC_PLANT_ROPE_INTERLEAVED", "ORC_PLANT_ROPE_FREQ",
          "ORC_PLANT_ROPE_SIGN"]


def test_unplanted_oracle_passes_the_pins():
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        str(ROOT / "tests" / "test_oracle_pins.py")],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("plant", PLANTS)
def test_pins_catch_planted_mistake(plant):
    env = dict(os.environ, ORACLE_PLANT=plant)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        str(ROOT / "tests" / "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"no pin failed with {plant}"
    assert "failed" in r.stdout
