"""CPU oracle for the batch-1 decode step (test infrastructure only; see oracle.cpp)."""
