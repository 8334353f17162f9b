"""CPU oracle for the DSA indexer hot path.  Test infrastructure only: imported by
tests, the smoke check and the benchmark's CPU-baseline leg, never by the library."""
