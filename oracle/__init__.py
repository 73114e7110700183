"""CPU oracle of the MoE expert block: test infrastructure, never the product path."""
