"""fp64 CPU oracle of the LongFlow fused decode step.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
CPU-baseline / reference leg of bench.py.  The product path never imports it.
"""
from .longflow_oracle import (OracleSequence, OracleUnit, Policy, StepResult, attention,
                              choose_victim, group_step, longflow_scores, value_norm)

__all__ = ["OracleSequence", "OracleUnit", "Policy", "StepResult", "attention", "choose_victim",
           "group_step", "longflow_scores", "value_norm"]
