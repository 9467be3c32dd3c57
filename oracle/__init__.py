"""CPU oracle of the GDN core forward (test infrastructure only)."""
