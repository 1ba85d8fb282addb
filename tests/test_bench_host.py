"""bench.py host logic that needs no GPU: plan overrides given with --tune are set
through ssm_tuning_set, recorded in the printed line's config, and malformed ones are
rejected before anything runs."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from selective_state_space_143_b300 import _lib  # noqa: E402


@pytest.fixture(autouse=True)
def _restore():
    yield
    bench.TUNING.clear()
    for k in (_lib.SSM_TUNE_DIAG_EXP_POLY, _lib.SSM_TUNE_BWD_PARTS):
        _lib.tuning_set(k, 0)


def test_tune_sets_the_knob_and_the_line_records_it(capsys):
    bench.apply_tuning(["DIAG_EXP_POLY=1", "bwd_parts=12"])
    assert _lib.tuning_get(_lib.SSM_TUNE_DIAG_EXP_POLY) == 1
    assert _lib.tuning_get(_lib.SSM_TUNE_BWD_PARTS) == 12
    bench.emit({"metric": "m", "config": {"workload": "w"}})
    line = json.loads(capsys.readouterr().out.strip())
    assert line["config"]["tuning"] == {"SSM_TUNE_DIAG_EXP_POLY": 1, "SSM_TUNE_BWD_PARTS": 12}


def test_no_tune_leaves_the_config_alone(capsys):
    bench.emit({"metric": "m", "config": {"workload": "w"}})
    assert "tuning" not in json.loads(capsys.readouterr().out.strip())["config"]


@pytest.mark.parametrize("spec", ["NO_SUCH_KNOB=1", "DIAG_EXP_POLY", "DIAG_EXP_POLY=x"])
def test_malformed_tune_is_rejected(spec):
    with pytest.raises(SystemExit):
        bench.apply_tuning([spec])
    assert _lib.tuning_get(_lib.SSM_TUNE_DIAG_EXP_POLY) == 0
