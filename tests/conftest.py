import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def to_numpy(t):
    """torch tensor -> numpy; bf16 goes through fp32 (exact)."""
    import torch

    if t is None:
        return None
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        t = t.to(torch.float32)
    return t.numpy()


def oracle_inputs(inp):
    """synth.DecodeInputs -> oracle.decode.StepInputs (plain arrays)."""
    from oracle.decode import StepInputs

    return StepInputs(
        q=to_numpy(inp.q), k_pool=to_numpy(inp.k_pool), v_pool=to_numpy(inp.v_pool),
        k_scale=to_numpy(inp.k_scale), v_scale=to_numpy(inp.v_scale),
        page_table=to_numpy(inp.page_table), seq_lens=to_numpy(inp.seq_lens),
        proj=to_numpy(inp.proj),
    )


def oracle_params(w, selector=None):
    from oracle.decode import StepParams

    return StepParams(
        page_size=w.page_size, n_sel=w.n_sel_pages, n_sink=w.n_sink, n_recent=w.n_recent,
        selector=selector or w.selector, head_dim=w.head_dim, meta_dtype=w.q_dtype,
    )


@pytest.fixture
def rng():
    return np.random.default_rng(12345)
