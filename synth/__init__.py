"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This package only draws random numbers and describes workloads symbolically.
It holds none of the attention arithmetic: no mask evaluation, no tile
classification, no softmax.
"""
from .inputs import (  # noqa: F401
    WORKLOADS,
    Workload,
    MaskProgram,
    doc_lengths,
    doc_ids_from_lengths,
    make_doc_ids,
    make_qkv,
    make_alibi_slopes,
    make_workload_inputs,
)
