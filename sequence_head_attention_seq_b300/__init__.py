"""Causal multi-head attention on the Ulysses sequence/head layout, for B300 (sm_103a)."""
