"""CPU oracle of one GPT-2 training step (plain C, built twice: float and
double).  TEST INFRASTRUCTURE ONLY: used by tests/, ``__graft_entry__`` and
bench.py's CPU-baseline leg; the CUDA package never imports it."""
