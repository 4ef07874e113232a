"""CPU oracle for the hyper-connection read (test infrastructure only)."""
