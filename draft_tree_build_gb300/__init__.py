"""GB300 (sm_103a) draft-tree hot path: top-K marginals, best-first tree with
an online budget controller, tree-masked GQA attention and greedy verification,
behind the C ABI in ``include/bastion.h``.  ``bastion`` is the Python binding."""

__all__ = ["bastion"]
