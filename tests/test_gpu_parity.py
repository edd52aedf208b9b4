"""CUDA path vs the CPU oracle, element by element, through the C ABI."""
import numpy as np
import pytest
import torch

import synth
from synth import prompts as SP
from tests import _parity as PR

pytestmark = pytest.mark.gpu

TINY = synth.CONFIGS[1].model


@pytest.mark.parametrize("wdtype", ["f32", "bf16", "int4", "int4e3"])
def test_tiny_config_prefill_and_decode(gpu_lib, wdtype):
    """Config 1 (64 cached prompt tokens, 16 decode steps), and the same tiny
    model with bf16 and int4 linear layers, and with int3 experts in the int4
    model (int4e3).  The 64-token prompt runs through the chunked prefill's
    GEMMs, the decode steps through the decode kernel."""
    m = TINY.with_(wdtype="int4", expert_dtype="int3") if wdtype == "int4e3" else TINY.with_(wdtype=wdtype)
    rep = PR.run_single(m, prompt_len=64, n_decode=16)
    print(rep)
    assert not rep.failures, rep
    if wdtype == "f32":
        assert rep.max_x < 1e-4, rep


@pytest.mark.parametrize("prompt_len", [1, 2, 17, 127, 128, 129, 300])
def test_tiny_prompt_lengths_across_page_boundaries(gpu_lib, prompt_len):
    rep = PR.run_single(TINY, prompt_len=prompt_len, n_decode=3)
    assert not rep.failures, rep


def test_tiny_long_context_split_attention(gpu_lib):
    """A context long enough that attention splits into many chunks per head."""
    rep = PR.run_single(TINY.with_(wdtype="int4"), prompt_len=3000, n_decode=2, n_pages=64)
    assert not rep.failures, rep
