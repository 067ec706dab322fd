"""Parity of the CUDA library with the float64 oracle at the configurations' full sizes: the object
scene (100k Gaussians, 800x800), the outdoor scene (1.6M, 1297x840), one view of the large scene
(3M, 1959x1090, about 180M duplicates) and the contention scene (50k large Gaussians, 3840x2160).
The tiny scene (2k, 128x128) is already at its full size in the stage tests.

Each configuration runs in the launch configuration the benchmark times: the library defaults
(ADAPTIVE accumulation with its default threshold, bulk staging), plus the DIRECT backward. Stage
by stage (both sides take the oracle's preprocess outputs rounded to float32) at the parity bars,
then the whole step end to end (each side computes its own records). On the outdoor scene the step
also runs as the captured CUDA graph the benchmark replays, against the oracle.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from differentiable_gaussian_splatting_gs_gb300 import _abi, api  # noqa: E402

import _gpu_checks as gc  # noqa: E402
from _cases import full_size  # noqa: E402

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(autouse=True)
def _no_device_errors():
    yield
    assert api.gs_device_error() == _abi.GS_OK, "device error word set"


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_full_size_stages_match_oracle(cfg):
    d = full_size(cfg)
    s, cam = d["scene"], d["cam"]
    params = gc.dev_params(s)
    gc.check_preprocess(s, cam, d["pre"], params=params)
    proj = gc.dev_proj(d["rec"])
    opt = api.make_options(s.sh_degree)
    b = gc.check_bin(proj, cam, opt, d["vals"], d["ranges"])
    img, tf, nc = gc.check_fwd(proj, b, cam, opt, d["fwd"], d["stats"]["pairs_evaluated"])
    for mode in ("adaptive", "direct"):
        gc.check_bwd(proj, b, cam, api.make_options(s.sh_degree, bwd_mode=mode), tf, nc, d["dl_masked"],
                     d["grad2d_masked"])
    gc.check_preprocess_bwd(s, cam, d["pre"], d["grad2d32"], d["grads"], params=params)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_full_size_step_matches_oracle(cfg):
    d = full_size(cfg)
    gc.end_to_end(d["scene"], 0, pre=d["pre"], bins=d["bins"])


def test_full_size_graph_replay_matches_oracle():
    """The outdoor step captured into one CUDA graph (non-synchronising sort, programmatic
    launches) and replayed, with the oracle's upstream gradient, against the oracle."""
    d = full_size(2)
    gc.end_to_end(d["scene"], 0, pre=d["pre"], bins=d["bins"], graph=True)
