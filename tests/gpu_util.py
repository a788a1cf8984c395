"""Helpers shared by the GPU tests: run the CUDA path and the oracle on the
same seeded host inputs."""
import numpy as np
import torch

import oracle
from fp8_bit_attention_gb300 import workloads as W

TOL_REL_L2 = 5e-3


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def inputs(B, H, S, seed, **kw):
    return W.generate(W.custom(B, H, S, seed=seed, **kw))


def oracle_prep(q, k, v):
    return oracle.Prepared(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v))


def to_dev(*xs):
    return tuple(x.cuda() for x in xs)
