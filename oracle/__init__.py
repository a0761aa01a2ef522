"""CPU oracle of the SKV v1 format (test infrastructure; see oracle/README.md)."""
