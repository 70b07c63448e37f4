"""The settings the pages print (tests/golden/dspark_settings.txt, each with its
page and section) are the ones the oracle, the binding's defaults and the
workload shapes use."""
import inspect
import os

from oracle import loss as L
from serving_draft_verify_gb300 import _binding as bnd
from serving_draft_verify_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dspark_settings.txt")


def _settings():
    out = {}
    with open(GOLDEN) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                name, value = line.split()[:2]
                out[name] = float(value)
    return out


def test_loss_weights_and_decay():
    s = _settings()
    assert (L.ALPHA_CE, L.ALPHA_L1, L.ALPHA_CONF) == (s["ce_loss_alpha"], s["l1_loss_alpha"],
                                                      s["confidence_head_alpha"])
    assert L.DECAY_GAMMA == s["loss_decay_gamma"]
    p = inspect.signature(bnd.dspark_training_loss).parameters
    assert (p["alpha_ce"].default, p["alpha_l1"].default, p["alpha_conf"].default) == (
        s["ce_loss_alpha"], s["l1_loss_alpha"], s["confidence_head_alpha"])


def test_shapes():
    s = _settings()
    for cfg in (wl.QWEN3_8B, wl.DRAFT_27B):
        assert cfg.gamma == s["block_size"] and cfg.r == s["markov_rank"]
    assert wl.DRAFT_27B.H == s["hidden_size_27b"]
    assert wl.LOSS_BLOCK == s["training_block_size"]
