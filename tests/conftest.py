import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402
from oracle import dflash_oracle as O  # noqa: E402


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: minutes of CPU time")


def oracle_shape(s: synth.ModelShape) -> O.Shape:
    return O.Shape(s.n_layers, s.hidden, s.n_q, s.n_kv, s.head_dim, s.ffn, s.vocab, s.rope_theta, s.eps)


def _layers(w, prefix, n):
    out = []
    for i in range(n):
        p = f"{prefix}{i}."
        out.append(O.Layer(*(w[p + part] for part in synth.LAYER_PARTS)))
    return out


def oracle_models(wl: synth.Workload, w: dict):
    """Oracle Target/Draft objects from canonical host weights."""
    t = wl.target
    tg = O.Target(oracle_shape(t), w["embed"], _layers(w, "layers.", t.n_layers), w["final_norm"],
                  w["lm_head"], tuple(O.layer_indices(t.n_layers)))
    dr = O.Draft(oracle_shape(wl.draft), w["draft.w_fc"], w["draft.fc_norm"],
                 _layers(w, "draft.layers.", wl.draft_layers), w["draft.final_norm"], t.vocab - 1)
    return tg, dr


def shrink(wl: synth.Workload, **kw) -> synth.Workload:
    """A copy of a workload with some target fields or run fields replaced."""
    import dataclasses

    tfields = {k: v for k, v in kw.items() if k in synth.ModelShape.__dataclass_fields__}
    rfields = {k: v for k, v in kw.items() if k not in tfields}
    t = dataclasses.replace(wl.target, **tfields)
    return dataclasses.replace(wl, target=t, **rfields)


@pytest.fixture(scope="session")
def tiny():
    wl = synth.WORKLOADS["tiny-f32"]
    w = synth.host_weights(wl.target, wl.draft_layers, wl.dtype)
    return wl, w


@pytest.fixture(scope="session")
def rng():
    return np.random.default_rng(12345)
