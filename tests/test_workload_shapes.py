"""The workload shapes are pinned to the adapter counts the pages print
(xingyuzhitong.com "Fine-Tuning Memory Requirements", section "LoRA: freeze
the base, train small adapters")."""
import json
import os

from bit_quantized_lora_double_b300 import synth

FIG = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")))


def test_llama8b_layer_adapter_count():
    s = sum(n + k for _, n, k in synth.LLAMA8B_LAYER)
    assert s == FIG["llama31_8b_lora_sum_per_layer"]["value"]
    assert 16 * s == FIG["llama31_8b_lora_params_r16_per_layer"]["value"]
    g = FIG["llama31_8b_lora_params_r16_32_layers_millions"]
    assert abs(16 * s * g["layers"] / 1e6 - g["value"]) <= g["tolerance"]


def test_llama70b_layer_adapter_count():
    s = sum(n + k for _, n, k in synth.LLAMA70B_LAYER)
    g = FIG["llama_70b_lora_params_r16_millions"]
    assert abs(16 * s * g["layers"] / 1e6 - g["value"]) <= g["tolerance"]


def test_seeds_distinct():
    seeds = {synth.seed_for(w, t, p) for w in range(5) for t in synth.TENSOR for p in range(7)}
    assert len(seeds) == 5 * 5 * 7
