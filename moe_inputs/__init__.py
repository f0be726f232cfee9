"""Seeded synthetic inputs for the FP4 routed-MoE layer.

This module only draws random numbers and lays them out in the layer's
tensor formats. It holds none of the layer's arithmetic (no decoding,
routing, sorting or matrix products), so both the CPU oracle and the CUDA
path can consume its output without sharing any of the method.
"""
from .synth import CONFIGS, LayerInputs, make_config, make_gate_weights, make_layer, routing_sample_tokens

__all__ = ["CONFIGS", "LayerInputs", "make_config", "make_gate_weights", "make_layer", "routing_sample_tokens"]
