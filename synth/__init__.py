"""Seeded synthetic inputs shared by the tests, the oracle checks and the bench.

Holds the counter-based generators and the tree shapes only; nothing of the
attention method itself.
"""
from . import rng, trees  # noqa: F401
from .trees import (Workload, tiny_two_level, document_qa, few_shot, speculative,  # noqa: F401
                    tree_of_thought, flat_control, random_tree, grow_query_nodes, source_rows,
                    speculative_next_step, CONFIGS)
