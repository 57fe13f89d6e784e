"""fp64 CPU oracle of the Gated DeltaNet layer. Test infrastructure only."""
