"""CPU oracle of the SKV v1 format. Test infrastructure: only the tests, the
smoke check and the benchmark's CPU-baseline leg load it; the CUDA library
never imports it and shares no code with it."""
