"""fp64 CPU oracle for the GQA attention hot path -- test infrastructure only."""
